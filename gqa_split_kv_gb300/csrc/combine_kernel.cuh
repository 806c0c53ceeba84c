// Log-sum-exp combine of split partials into the bf16 output.
//
// For one (b, h): M = max_j m_j over live slots, w_j = exp(m_j - M),
// out = sum_j w_j acc_j / sum_j w_j l_j, in ascending j (the fixed merge order of
// "perf(qwen3.8): split the flash-decode KV range across warp-groups", section
// "Mechanism"; the partial/merge split of AstrAI commit 988e013 "csrc", split-KV
// items).  Each thread owns 4 consecutive output columns; D / 4 threads per row.
//
// Two modes:
//   planned:  called after the split kernel (programmatic dependent launch); the
//             piece count of each row comes from the split plan: rows with one
//             piece were written by the split kernel, rows of empty sequences are
//             written as zeros.
//   plain:    all S slots of every row, skipping slots with l == 0.
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
  static constexpr int NTHREADS = 128;
  static constexpr int TPR = D / 4;                  // threads per row
  static constexpr int RPC = NTHREADS / TPR;         // rows per CTA
};

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  using Cg = CombineGeo<D>;
  extern __shared__ int csmem[];
  int* lens = csmem;
  int* P = csmem + p.B;
  Plan pl{};
  if (p.planned) {
    // seq_lens is not written by the split kernel: read it before waiting.
    build_plan_arrays(p.seq_lens, p.B, p.max_len, lens, P);
    pl = make_plan(p.B, p.U, p.S, P);
  }
  pdl_wait_primary();

  const long long row = (long long)blockIdx.x * Cg::RPC + threadIdx.x / Cg::TPR;
  const int c4 = threadIdx.x % Cg::TPR;
  if (row >= (long long)p.B * p.Hq) return;
  const int b = (int)(row / p.Hq);
  const int h = (int)(row % p.Hq);
  int n = p.S;
  if (p.planned) {
    const int gi = h % p.G;
    const int u = (h / p.G) * p.ng + gi / p.gr;
    n = segment_pieces(pl, lens, P, b, u);
    if (n == 1) return;  // written directly by the split kernel
  }
  const float* ml = p.part_ml + (size_t)row * p.S * 2;
  const float4* acc = reinterpret_cast<const float4*>(p.part_acc + (size_t)row * p.S * D) + c4;
  const float kNegInf = -__int_as_float(0x7f800000);
  float M = kNegInf;
  for (int j = 0; j < n; ++j) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * j);
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int j = 0; j < n; ++j) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * j);
    if (v.y > 0.f) {
      const float w = expf(v.x - M);
      const float4 a = acc[(size_t)j * (D / 4)];
      num.x += w * a.x;
      num.y += w * a.y;
      num.z += w * a.z;
      num.w += w * a.w;
      den += w * v.y;
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint2 o;
  o.x = pack_bf16x2(num.x * inv, num.y * inv);
  o.y = pack_bf16x2(num.z * inv, num.w * inv);
  *reinterpret_cast<uint2*>(p.out + (size_t)row * D + 4 * c4) = o;
}

}  // namespace da
