// Host side of the causal prefill entry points (declared in include/decode_attn.h):
// argument checks, TMA maps of the caller's cache and the launch of the prefill
// kernel.  Part of the library's single translation unit (included at the end of
// decode_attn.cu, after its helpers).
#pragma once

#include "prefill_kernel.cuh"
#include "prefill_tc.cuh"

namespace da {
namespace {

template <int D, bool PAGED>
int launch_prefill(const PrefillParams& prm, unsigned grid, int dev, cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {false};
  auto kern = prefill_kernel<D, PAGED>;
  const int smem = PrefillGeo<D>::SMEM;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        cudaGetLastError();
        return DA_ERR_UNSUPPORTED;
      }
      attr_done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PrefillGeo<D>::NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

template <int D, bool PAGED>
int launch_prefill_tc(const PrefillParams& prm, unsigned grid, int dev, cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {false};
  auto kern = prefill_tc_kernel<D, PAGED>;
  using Gm = PrefillTcGeo<D>;
  const int smem = Gm::SMEM;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        cudaGetLastError();
        return DA_ERR_UNSUPPORTED;
      }
      if (Gm::NQT == 2) {
        // the softmax warpgroups raise their registers (setmaxnreg.inc) out of what
        // the launch gave the CTA; a build whose per-thread count is below the
        // split would wait there for ever, so it is refused instead
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
          cudaGetLastError();
          return DA_ERR_CUDA;
        }
        if (fa.numRegs * Gm::NTHREADS < Gm::REG_POOL_NEEDED) return DA_ERR_UNSUPPORTED;
      }
      attr_done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PrefillTcGeo<D>::NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

// Keys per tile of the tensor-core kernel (head_dim 64, 128, 256); 0: head_dim 32
// runs the warp-MMA kernel.
int tc_tile_keys(int D) {
  return D == 64 ? PrefillTcGeo<64>::BK : D == 128 ? PrefillTcGeo<128>::BK : D == 256 ? PrefillTcGeo<256>::BK : 0;
}
int tc_query_tiles(int D) {
  return D == 64 ? PrefillTcGeo<64>::NQT : D == 128 ? PrefillTcGeo<128>::NQT : PrefillTcGeo<256>::NQT;
}

// Shared by the contiguous and paged calls.  max_len: lengths are clamped to it
// (max_ctx, or min(max_pages * page_size, max_seq_len)).
int prefill_call(bool paged, const void* q, const void* k, const void* v, const int* page_table, const int* seq_lens,
                 int B, int q_len, int Hq, int Hkv, int D, int max_len, int page_size, int max_pages, int num_pages,
                 float scale, void* out, void* stream) {
  if (B < 0 || q_len < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !std::isfinite(scale)) return DA_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128 && D != 256) return DA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G > 64) return DA_ERR_UNSUPPORTED;  // one token's G rows must fit a CTA (64 or 128 rows)
  if ((long long)q_len * Hq > (1LL << 28)) return DA_ERR_UNSUPPORTED;
  if (B == 0 || q_len == 0) return DA_OK;
  if (!q || !out || !aligned(q, 16) || !aligned(out, 16)) return DA_ERR_INVALID_ARG;
  const int tcbk = tc_tile_keys(D);
  // query tokens per CTA: a whole number of tokens per 128-row query tile (the
  // tensor-core kernel has one or two such tiles), or per the warp-MMA kernel's rows
  const int BQ = tcbk ? tc_query_tiles(D) * (PrefillTcGeo<128>::M / G) : PrefillGeo<32>::ROWS / G;
  const long long nqb = (q_len + BQ - 1) / BQ;
  if (nqb * B * Hkv > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_bytes = (size_t)B * q_len * Hq * D * 2;
  if (max_len == 0 || (paged && num_pages == 0)) {
    if (cudaMemsetAsync(out, 0, out_bytes, st) != cudaSuccess) {
      cudaGetLastError();
      return DA_ERR_CUDA;
    }
    return DA_OK;
  }
  if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return DA_ERR_INVALID_ARG;
  int dev, sms, smem_optin;
  if (current_device(&dev) || device_info(dev, &sms, &smem_optin)) return DA_ERR_CUDA;

  PrefillParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const int SW = sub_width(D);
  const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
  if (!paged) {
    // the decode cache map with boxes of a whole tile: [D/SW][keys][SW] (64 keys for
    // the warp-MMA kernel, BK for the tensor-core kernel)
    const cuuint64_t dims[5] = {(cuuint64_t)SW, (cuuint64_t)max_len, (cuuint64_t)(D / SW), (cuuint64_t)Hkv,
                                (cuuint64_t)B};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW * 2, (cuuint64_t)D * 2, row * (cuuint64_t)max_len};
    const cuuint32_t box[5] = {(cuuint32_t)SW, (cuuint32_t)(tcbk ? tcbk : PrefillGeo<32>::BK), (cuuint32_t)(D / SW),
                               1, 1};
    if (int e = encode_map(&prm.tm_k, k, 5, dims, strides, box, D)) return e;
    if (int e = encode_map(&prm.tm_v, v, 5, dims, strides, box, D)) return e;
    prm.box_shift = 2;
  } else {
    // boxes of R rows of one page (R = 64, 32 or 16, dividing the page size); the
    // tensor-core kernel copies one swizzle column per box, so its tile is
    // [D/SW][keys][SW] like the contiguous one
    const int box_shift = page_size % 64 == 0 ? 2 : page_size % 32 == 0 ? 1 : 0;
    const cuuint64_t dims[5] = {(cuuint64_t)SW, (cuuint64_t)page_size, (cuuint64_t)(D / SW), (cuuint64_t)Hkv,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW * 2, (cuuint64_t)D * 2, row * (cuuint64_t)page_size};
    const cuuint32_t box[5] = {(cuuint32_t)SW, (cuuint32_t)(16 << box_shift), (cuuint32_t)(tcbk ? 1 : D / SW), 1, 1};
    if (int e = encode_map(&prm.tm_k, k, 5, dims, strides, box, D)) return e;
    if (int e = encode_map(&prm.tm_v, v, 5, dims, strides, box, D)) return e;
    prm.box_shift = box_shift;
  }
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.seq_lens = seq_lens;
  prm.page_table = page_table;
  prm.B = B;
  prm.q_len = q_len;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = G;
  prm.BQ = BQ;
  prm.nqb = (int)nqb;
  {
    // launch groups of (b, h) units whose K/V (bf16 K + V of max_len tokens) fit in
    // about 48 MB of L2 together
    const long long unit_bytes = 4LL * D * (max_len > 0 ? max_len : 1);
    long long g = (48LL << 20) / unit_bytes;
    g = g < 1 ? 1 : g;
    prm.grp = (int)(g < (long long)B * Hkv ? g : (long long)B * Hkv);
  }
  prm.max_len = max_len;
  prm.page_size = paged ? page_size : 0;
  prm.max_pages = paged ? max_pages : 0;
  prm.num_pages = paged ? num_pages : 0;
  prm.page_shift = paged && (page_size & (page_size - 1)) == 0 ? __builtin_ctz((unsigned)page_size) : -1;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.timeout_ns = kWaitTimeoutNs;
  const unsigned grid = (unsigned)(nqb * B * Hkv);
  switch (D) {
    case 32: return paged ? launch_prefill<32, true>(prm, grid, dev, st) : launch_prefill<32, false>(prm, grid, dev, st);
    case 64:
      return paged ? launch_prefill_tc<64, true>(prm, grid, dev, st) : launch_prefill_tc<64, false>(prm, grid, dev, st);
    case 128:
      return paged ? launch_prefill_tc<128, true>(prm, grid, dev, st) : launch_prefill_tc<128, false>(prm, grid, dev, st);
    default:
      return paged ? launch_prefill_tc<256, true>(prm, grid, dev, st) : launch_prefill_tc<256, false>(prm, grid, dev, st);
  }
}

}  // namespace
}  // namespace da

extern "C" int prefill_attn_contig(const void* q, const void* k, const void* v, const int* seq_lens, int batch,
                                   int q_len, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx, float scale,
                                   void* out, void* stream) {
  if (max_ctx < 0) return DA_ERR_INVALID_ARG;
  return prefill_call(false, q, k, v, nullptr, seq_lens, batch, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx, 0, 0, 0,
                      scale, out, stream);
}

extern "C" int prefill_attn_paged(const void* q, const void* k_pool, const void* v_pool, const int* page_table,
                                  const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim, int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                                  float scale, void* out, void* stream) {
  if (page_size <= 0 || max_pages_per_seq < 0 || num_pages < 0 || max_seq_len < 0) return DA_ERR_INVALID_ARG;
  if (page_size % 16 != 0) return DA_ERR_UNSUPPORTED;
  if (batch > 0 && q_len > 0 && (!seq_lens || !page_table || !aligned(page_table, 4))) return DA_ERR_INVALID_ARG;
  long long cap = (long long)max_pages_per_seq * page_size;
  if (cap > max_seq_len) cap = max_seq_len;
  if (cap > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  return prefill_call(true, q, k_pool, v_pool, page_table, seq_lens, batch, q_len, num_q_heads, num_kv_heads,
                      head_dim, (int)cap, page_size, max_pages_per_seq, num_pages, scale, out, stream);
}
