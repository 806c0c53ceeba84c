// Log-sum-exp combine of split partials into the bf16 output.
//
// For one (b, h): M = max_j m_j over live slots (l_j > 0), w_j = exp(m_j - M),
// out = sum_j w_j acc_j / sum_j w_j l_j (the merge of "perf(qwen3.8): split the
// flash-decode KV range across warp-groups", section "Mechanism"; the
// partial/merge split of AstrAI commit 988e013 "csrc", split-KV items).
//
// One CTA per row at a time (grid-strided over rows).  All (m, l) of the row are
// loaded at once and reduced to M and the weights in shared memory; the slot x
// column products are spread over the 256 threads (JL slot lanes x D/4 column
// groups of 4), so every load of a row is in flight together; the JL lane sums
// are added in ascending lane order.  The summation order is fixed, so results
// are bitwise reproducible.
//
// Two modes:
//   planned:  after the split kernel (programmatic dependent launch); a row's slot
//             count is its segment's piece count under the split plan; rows with one
//             piece were written by the split kernel, rows of empty sequences are
//             written as zeros.
//   plain:    every S slot of every row, skipping slots with l == 0.
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
  int G, U, ng, gr, max_len;
};

template <int D>
struct CombineGeo {
  static constexpr int NTHREADS = 256;
  static constexpr int TPS = D / 4;               // threads per slot (4 columns each)
  static constexpr int JL = NTHREADS / TPS;       // slot lanes
  // shared: plan arrays (2B+1 ints) | weights, l (S floats each) | lane sums (NTHREADS float4) | misc
  static int smem_bytes(int B, int S, bool planned) {
    return ((planned ? (2 * B + 1) * 4 : 0) + 15) / 16 * 16 + 2 * (((S * 4 + 15) / 16) * 16) + NTHREADS * 16 + 64;
  }
};

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
  using Cg = CombineGeo<D>;
  extern __shared__ __align__(16) uint8_t csm[];
  int* lens = reinterpret_cast<int*>(csm);
  int* P = lens + p.B;
  const int plan_bytes = p.planned ? (2 * p.B + 1) * 4 : 0;
  float* wts = reinterpret_cast<float*>(csm + ((plan_bytes + 15) / 16) * 16);
  float* lsm = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(wts) + ((p.S * 4 + 15) / 16) * 16);
  float4* lane_sum = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(lsm) + ((p.S * 4 + 15) / 16) * 16);
  float* red = reinterpret_cast<float*>(lane_sum + Cg::NTHREADS);  // [0..7] warp maxima, [8] M, [9] den

  Plan pl{};
  if (p.planned) {
    // seq_lens is not written by the split kernel: read it before waiting on it.
    build_plan_arrays(p.seq_lens, p.B, p.max_len, lens, P);
    pl = make_plan(p.B, p.U, p.S, P);
  }
  pdl_wait_primary();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int jl = tid / Cg::TPS, c4 = tid % Cg::TPS;
  const float kNegInf = -__int_as_float(0x7f800000);
  const long long rows = (long long)p.B * p.Hq;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = (int)(row / p.Hq);
    const int h = (int)(row % p.Hq);
    int n = p.S;
    if (p.planned) {
      const int u = (h / p.G) * p.ng + (h % p.G) / p.gr;
      n = segment_pieces(pl, lens, P, b, u);
      if (n == 1) continue;  // written directly by the split kernel
    }
    const float* ml = p.part_ml + (size_t)row * p.S * 2;
    // 1. M over live slots
    float mloc = kNegInf;
    for (int j = tid; j < n; j += Cg::NTHREADS) {
      const float2 v = *reinterpret_cast<const float2*>(ml + 2 * j);
      wts[j] = v.y > 0.f ? v.x : kNegInf;
      lsm[j] = v.y > 0.f ? v.y : 0.f;
      if (v.y > 0.f) mloc = fmaxf(mloc, v.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if (lane == 0) red[warp] = mloc;
    __syncthreads();
    if (tid == 0) {
      float M = red[0];
      for (int w = 1; w < Cg::NTHREADS / 32; ++w) M = fmaxf(M, red[w]);
      red[8] = M;
    }
    __syncthreads();
    const float M = red[8];
    // 2. weights w_j = exp(m_j - M) (0 for dead slots); den = sum_j w_j l_j in ascending j
    for (int j = tid; j < n; j += Cg::NTHREADS) {
      const float mj = wts[j];
      wts[j] = mj == kNegInf ? 0.f : expf(mj - M);
    }
    __syncthreads();
    if (tid == 0) {
      float den = 0.f;
      for (int j = 0; j < n; ++j) den += wts[j] * lsm[j];
      red[9] = den;
    }
    // 3. weighted column sums, slots strided over the JL lanes
    const float4* acc = reinterpret_cast<const float4*>(p.part_acc + (size_t)row * p.S * D) + c4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = jl; j < n; j += Cg::JL) {
      const float w = wts[j];
      const float4 a = acc[(size_t)j * (D / 4)];
      s.x += w * a.x;
      s.y += w * a.y;
      s.z += w * a.z;
      s.w += w * a.w;
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
      const float den = red[9];
      const float inv = den > 0.f ? 1.f / den : 0.f;
      uint2 o;
      o.x = pack_bf16x2(t.x * inv, t.y * inv);
      o.y = pack_bf16x2(t.z * inv, t.w * inv);
      *reinterpret_cast<uint2*>(p.out + (size_t)row * D + 4 * c4) = o;
    }
    __syncthreads();
  }
}

}  // namespace da
