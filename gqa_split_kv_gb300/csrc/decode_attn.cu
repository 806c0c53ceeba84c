// C-ABI entry points of the decode-attention library (declared in include/decode_attn.h).
//
// Host side of every call: validate the arguments, build the TMA tensor maps of
// the caller's K/V/Q buffers and enqueue the persistent split kernel, which also
// merges segments cut into at most 8 pieces.
// When the plan allows longer segments, the combine kernel follows as a
// programmatic dependent launch (its CTAs start while the split kernel drains and
// wait on the device for it) and merges those.  decode_combine runs the
// stand-alone merge.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/decode_attn.h"
#include "combine_kernel.cuh"
#include "split_kernel.cuh"

namespace da {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per bounded wait

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
std::atomic<unsigned int> g_epoch{0};

// A fresh non-zero tag for the per-segment counters of one call.
unsigned int next_epoch() {
  unsigned int e = ++g_epoch;
  while (e == 0) e = ++g_epoch;
  return e;
}
int g_num_sms[kMaxDevices] = {0};
int g_smem_optin[kMaxDevices] = {0};

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? DA_OK : DA_ERR_CUDA; }

int device_info(int dev, int* sms, int* smem_optin) {
  if (dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_num_sms[dev] == 0) {
    int s = 0, m = 0;
    if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return DA_ERR_CUDA;
    }
    g_num_sms[dev] = s;
    g_smem_optin[dev] = m;
  }
  *sms = g_num_sms[dev];
  *smem_optin = g_smem_optin[dev];
  return DA_OK;
}

int get_encoder(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr) {
      cudaGetLastError();
      return DA_ERR_CUDA;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = g_encode;
  return DA_OK;
}

// Tiled map; dims/box innermost first, strides in bytes for dims 1..rank-1.
int encode_map_t(CUtensorMap* m, CUtensorMapDataType type, CUtensorMapSwizzle swz, const void* base, int rank,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn enc;
  if (int st = get_encoder(&enc)) return st;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_INVALID_ARG;
}

// Tiled bf16 map with the swizzle the kernels read (128-byte rows, 64-byte at D = 32).
int encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, int head_dim) {
  return encode_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      head_dim >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, base, rank, dims,
                      strides, box);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int sub_width(int D) { return D >= 64 ? 64 : 32; }
// int8 tiles: bytes per swizzle row and the swizzle the kernels read
int sub_width8(int D) { return D >= 128 ? 128 : D; }
CUtensorMapSwizzle swizzle8(int D) { return D >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE; }

// tokens per tile of the split kernel for a contiguous cache of head_dim D and the
// cache's element type (the TMA box height; the kernel's expected byte count uses
// the same geometry)
int tile_tokens(int D, bool kv8) {
  switch (D) {
    case 32: return kv8 ? SplitGeo<32, 1, true>::T : SplitGeo<32>::T;
    case 64: return kv8 ? SplitGeo<64, 1, true>::T : SplitGeo<64>::T;
    case 128: return kv8 ? SplitGeo<128, 1, true>::T : SplitGeo<128>::T;
    default: return kv8 ? SplitGeo<256, 1, true>::T : SplitGeo<256>::T;
  }
}

// Query heads of one KV head are processed in ceil(G / 8) equal sub-groups.
void head_groups(int G, int* ng, int* gr) {
  *ng = (G + 7) / 8;
  *gr = (G + *ng - 1) / *ng;
}

// Sub-groups per pass over a KV head: the largest power of two, up to what the
// shared memory holds, that divides the sub-group count (no warp group sits
// idle in a pass); npass passes per KV head.
void group_passes(int ng, int D, int* ngp, int* npass) {
  const int cap = D == 128 ? SplitGeo<128>::NGP_MAX : D == 256 ? SplitGeo<256>::NGP_MAX
                : D == 64 ? SplitGeo<64>::NGP_MAX : SplitGeo<32>::NGP_MAX;
  int g = 1;
  while (g * 2 <= cap && ng % (g * 2) == 0) g *= 2;
  *ngp = g;
  *npass = ng / g;
}

// Offset of the plan arrays in the split kernel's shared memory for a geometry;
// the kernel needs OFF_PLAN + (2 B + 2) * 4 + 1024 bytes (SplitGeo::smem_bytes).
template <int D, bool PG, bool KV8>
int plan_offset_t(int ngp) {
  if (ngp == 1) return SplitGeo<D, 1, KV8, PG>::OFF_PLAN;
  if (ngp == 2) return SplitGeo<D, 2, KV8, PG>::OFF_PLAN;
  if constexpr (SplitGeo<D>::NGP_MAX >= 4) return SplitGeo<D, 4, KV8, PG>::OFF_PLAN;
  return 1 << 30;
}

template <int D>
int plan_offset_d(bool paged, bool kv8, int ngp) {
  return paged ? (kv8 ? plan_offset_t<D, true, true>(ngp) : plan_offset_t<D, true, false>(ngp))
               : (kv8 ? plan_offset_t<D, false, true>(ngp) : plan_offset_t<D, false, false>(ngp));
}

// Largest batch whose plan fits the split kernel's shared memory (227 KB per CTA).
int max_batch_for(int D, bool paged, bool kv8, int ngp) {
  const int off = D == 32 ? plan_offset_d<32>(paged, kv8, ngp) : D == 64 ? plan_offset_d<64>(paged, kv8, ngp)
                : D == 128 ? plan_offset_d<128>(paged, kv8, ngp) : plan_offset_d<256>(paged, kv8, ngp);
  const int room = 227 * 1024 - 1024 - off;
  return room < 16 ? 0 : (room / 4 - 2) / 2;
}

struct Launch {
  int B, Hq, Hkv, D, max_len, S;  // Hq counts rows: query heads x qlen
  int qlen;
  float scale;
  const void* q;
  const int* seq_lens;
  const int* page_table;
  int page_size, max_pages, num_pages, box_shift;
  float* part_acc;
  float* part_ml;
  unsigned long long* seg_counters;
  void* out;
  cudaStream_t stream;
  bool paged;
  bool kv8;                           // int8 K/V with per-(token, KV head) scales
  const CUtensorMap* tks = nullptr;   // their scale maps
  const CUtensorMap* tvs = nullptr;
};

template <int D, bool PAGED, int NGP, bool KV8>
int launch_split_ngp(const SplitParams& prm, int grid, int smem_optin, int dev, cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {false};
  auto kern = split_kernel<D, PAGED, NGP, KV8>;
  const int smem = SplitGeo<D, NGP, KV8, PAGED>::smem_bytes(prm.B);
  if (smem > smem_optin || smem > 227 * 1024) return DA_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        cudaGetLastError();
        return DA_ERR_UNSUPPORTED;
      }
      attr_done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(SplitGeo<D, NGP, KV8, PAGED>::NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

// The split kernel is built for 1, 2 and 4 sub-groups per pass (up to NGP_MAX),
// for bf16 and for int8 caches.
template <int D, bool PAGED, bool KV8>
int launch_split_kv(const SplitParams& prm, int grid, int smem_optin, int dev, cudaStream_t st) {
  if (prm.ngp == 1) return launch_split_ngp<D, PAGED, 1, KV8>(prm, grid, smem_optin, dev, st);
  if (prm.ngp == 2) return launch_split_ngp<D, PAGED, 2, KV8>(prm, grid, smem_optin, dev, st);
  if constexpr (SplitGeo<D>::NGP_MAX >= 4) {
    if (prm.ngp == 4) return launch_split_ngp<D, PAGED, 4, KV8>(prm, grid, smem_optin, dev, st);
  }
  return DA_ERR_UNSUPPORTED;
}

template <int D, bool PAGED>
int launch_split(const SplitParams& prm, int grid, int smem_optin, int dev, cudaStream_t st, bool kv8) {
  return kv8 ? launch_split_kv<D, PAGED, true>(prm, grid, smem_optin, dev, st)
             : launch_split_kv<D, PAGED, false>(prm, grid, smem_optin, dev, st);
}

template <int D>
int launch_combine(const CombineParams& prm, int dev, int sms, cudaStream_t st, bool dependent) {
  static bool attr_done[kMaxDevices] = {false};
  auto kern = combine_kernel<D>;
  const int smem = CombineGeo<D>::smem_bytes(prm.B, prm.S, prm.planned != 0);
  if (smem > 227 * 1024) return DA_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        cudaGetLastError();
        return DA_ERR_UNSUPPORTED;
      }
      attr_done[dev] = true;
    }
  }
  // grid-strided over (row, column chunk) items; after the split kernel one CTA per SM, so every CTA
  // fits beside a split CTA, starts early and has its plan ready when the split
  // kernel completes; alone, a few CTAs per SM
  const long long items = (long long)prm.B * prm.Hq * CombineGeo<D>::NCH;
  const long long cap = (dependent ? 1LL : 4LL) * (sms > 0 ? sms : 1);
  const long long grid = items < cap ? items : cap;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(CombineGeo<D>::NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

template <int D>
int run_decode(const Launch& a, const CUtensorMap& tk, const CUtensorMap& tv, int dev, int sms, int smem_optin) {
  int ng, gr;
  head_groups(a.Hq / a.Hkv, &ng, &gr);
  int ngp, npass;
  group_passes(ng, D, &ngp, &npass);
  SplitParams prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.tm_k = tk;
  prm.tm_v = tv;
  {
    const int SW = sub_width(D);
    const cuuint64_t dims[4] = {(cuuint64_t)SW, (cuuint64_t)(D / SW), (cuuint64_t)a.Hq, (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {(cuuint64_t)SW * 2, (cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)SW, 1, (cuuint32_t)gr, 1};
    if (int st = encode_map(&prm.tm_q, a.q, 4, dims, strides, box, D)) return st;
  }
  prm.seq_lens = a.seq_lens;
  prm.page_table = a.page_table;
  prm.part_acc = a.part_acc;
  prm.part_ml = a.part_ml;
  prm.seg_counters = a.seg_counters;
  prm.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  prm.epoch = next_epoch();
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.G = a.Hq / a.Hkv;
  prm.ng = ng;
  prm.gr = gr;
  prm.ngp = ngp;
  prm.npass = npass;
  prm.U = a.Hkv * npass;
  prm.max_len = a.max_len;
  prm.qlen = a.qlen;
  prm.page_size = a.page_size;
  prm.max_pages = a.max_pages;
  prm.num_pages = a.num_pages;
  prm.box_shift = a.box_shift;
  prm.page_shift = -1;
  for (int s = 4; s < 31; ++s)
    if (a.page_size == (1 << s)) prm.page_shift = s;
  prm.S = a.S;
  // small contiguous batches (latency-bound calls): guessed first tiles before the plan
  prm.spec_first = !a.paged && a.B <= 4 ? 1 : 0;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.timeout_ns = kWaitTimeoutNs;

  // one persistent CTA per SM, never more CTAs than ranges or blocks of work
  const long long nblk_max = (a.max_len + kBlockTokens - 1) / kBlockTokens;
  if ((long long)a.B * prm.U * (nblk_max + 3 + plan_gap_blocks(D)) >= (1LL << 30) || (long long)a.B * a.Hq >= (1LL << 30))
    return DA_ERR_UNSUPPORTED;  // the device plan counts line positions in 32 bits
  long long ranges = a.S == 1 ? (long long)a.B * prm.U : (long long)(a.S - 1) * prm.U;
  const long long work = (long long)a.B * prm.U * (nblk_max > 0 ? nblk_max : 1);
  if (ranges > work) ranges = work;
  const int grid = (int)(ranges < sms ? ranges : sms);
  if (a.kv8) {
    prm.tm_ks = *a.tks;
    prm.tm_vs = *a.tvs;
  }
  if (int st = (a.paged ? launch_split<D, true>(prm, grid, smem_optin, dev, a.stream, a.kv8)
                        : launch_split<D, false>(prm, grid, smem_optin, dev, a.stream, a.kv8)))
    return st;
  if (a.S <= kFusedMergeMax) return DA_OK;  // every segment is merged inside the split kernel
  CombineParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.part_acc = a.part_acc;
  cp.part_ml = a.part_ml;
  cp.out = prm.out;
  cp.seq_lens = a.seq_lens;
  cp.B = a.B;
  cp.Hq = a.Hq;
  cp.S = a.S;
  cp.planned = 1;
  cp.G = prm.G;
  cp.U = prm.U;
  cp.ng = ng;
  cp.gr = gr;
  cp.ngp = ngp;
  cp.npass = npass;
  cp.max_len = a.max_len;
  return launch_combine<D>(cp, dev, sms, a.stream, true);
}

int check_common(const void* q, const void* out, int B, int Hq, int Hkv, int D, float scale, int S,
                 const float* part_acc, const float* part_ml, const unsigned long long* seg_counters) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return DA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DA_ERR_INVALID_ARG;
  if (S < 1 || S > DA_MAX_SPLITS) return DA_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128 && D != 256) return DA_ERR_UNSUPPORTED;
  if (Hq / Hkv > 64) return DA_ERR_UNSUPPORTED;
  if (B == 0) return DA_OK;
  if (!q || !out) return DA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return DA_ERR_INVALID_ARG;
  if (S >= 2) {
    if (!part_acc || !part_ml || !seg_counters) return DA_ERR_WORKSPACE;
    if (!aligned(part_acc, 16) || !aligned(part_ml, 8) || !aligned(seg_counters, 8)) return DA_ERR_INVALID_ARG;
  }
  return DA_OK;
}

int dispatch(const Launch& a, const CUtensorMap& tk, const CUtensorMap& tv, int dev, int sms, int smem_optin) {
  // the batch limit of the plan in shared memory (decode_max_batch)
  int ng, gr, ngp, npass;
  head_groups(a.Hq / a.Hkv, &ng, &gr);
  group_passes(ng, a.D, &ngp, &npass);
  if (a.B > max_batch_for(a.D, a.paged, a.kv8, ngp)) return DA_ERR_UNSUPPORTED;
  switch (a.D) {
    case 32: return run_decode<32>(a, tk, tv, dev, sms, smem_optin);
    case 64: return run_decode<64>(a, tk, tv, dev, sms, smem_optin);
    case 128: return run_decode<128>(a, tk, tv, dev, sms, smem_optin);
    default: return run_decode<256>(a, tk, tv, dev, sms, smem_optin);
  }
}

int zero_output(void* out, int B, int Hq, int D, cudaStream_t st) {
  if (cudaMemsetAsync(out, 0, (size_t)B * Hq * D * 2, st) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

}  // namespace
}  // namespace da

using namespace da;

extern "C" int decode_num_splits(int batch, int num_kv_heads, int max_seq_len, int head_dim, int num_sms) {
  if (batch < 0 || num_kv_heads <= 0 || max_seq_len < 0 || head_dim <= 0) return -DA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    int dev, smem;
    if (current_device(&dev) || device_info(dev, &num_sms, &smem)) return -DA_ERR_CUDA;
  }
  const long long nblk = ((long long)max_seq_len + kBlockTokens - 1) / kBlockTokens;
  if (nblk <= 1) return 1;
  long long S = (num_sms + num_kv_heads - 1) / num_kv_heads + 1;
  if (S > nblk) S = nblk;
  if (S > DA_MAX_SPLITS) S = DA_MAX_SPLITS;
  if (S < 2) S = 2;
  return (int)S;
}

extern "C" int decode_num_splits_multi(int batch, int q_len, int num_q_heads, int num_kv_heads, int max_seq_len,
                                       int head_dim, int num_sms) {
  if (q_len < 1 || q_len > DA_MAX_QLEN || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads * q_len > 64)
    return -DA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256) return -DA_ERR_UNSUPPORTED;
  int ng, gr, ngp, npass;
  head_groups(num_q_heads / num_kv_heads * q_len, &ng, &gr);
  group_passes(ng, head_dim, &ngp, &npass);
  return decode_num_splits(batch, num_kv_heads * npass, max_seq_len, head_dim, num_sms);
}

extern "C" int decode_plan_pieces(const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim, int max_len, int num_splits, int* records, int capacity, int* count) {
  if (!count) return DA_ERR_INVALID_ARG;
  *count = 0;
  if (batch < 0 || max_len < 0 || capacity < 0 || q_len < 1 || q_len > DA_MAX_QLEN || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || num_splits < 1 || num_splits > DA_MAX_SPLITS)
    return DA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256) return DA_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads * q_len;  // rows per KV head
  if (G > 64) return DA_ERR_UNSUPPORTED;
  const int B = batch, D = head_dim, S = num_splits;
  if (B == 0) return DA_OK;
  int ng, gr, ngp, npass;
  head_groups(G, &ng, &gr);
  group_passes(ng, D, &ngp, &npass);
  const int U = num_kv_heads * npass;
  const int gap = plan_gap_blocks(D);
  const long long nblk_max = ((long long)max_len + kBlockTokens - 1) / kBlockTokens;
  if ((long long)B * U * (nblk_max + 3 + gap) >= (1LL << 30)) return DA_ERR_UNSUPPORTED;
  // the arrays build_plan_arrays forms on the device
  std::vector<int> lens(B), P(B + 2);
  int run = 0, mx = 0;
  for (int b = 0; b < B; ++b) {
    int L = seq_lens ? seq_lens[b] : max_len;
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    lens[b] = L;
    P[b] = run;
    const int nb = (L + kBlockTokens - 1) / kBlockTokens;
    run += segment_width(nb, gap);
    mx = nb > mx ? nb : mx;
  }
  P[B] = run;
  P[B + 1] = mx;
  const Plan pl = make_plan(B, U, S, gap, P.data());
  // every range in order, with the walker the kernel's CTAs use
  PieceWalker walk;
  walk.init(0, 1);
  Piece pc;
  std::vector<int> rec;
  while (walk.next(pl, lens.data(), P.data(), B, true, pc)) {
    const int h = pc.u / npass, pass_u = pc.u % npass;
    const int nsg = ngp < ng - pass_u * ngp ? ngp : ng - pass_u * ngp;
    const int row0 = h * G + pass_u * ngp * gr;
    const int nrows = nsg * gr < G - pass_u * ngp * gr ? nsg * gr : G - pass_u * ngp * gr;
    const int fields[9] = {pc.b, row0, nrows, pc.j, pc.npieces, pc.t0, pc.t1, pc.t0, pc.t1};
    rec.insert(rec.end(), fields, fields + 9);
  }
  const int n = (int)(rec.size() / 9);
  // a segment written straight to the output leaves no partial; every other piece
  // leaves its own in slot j
  for (int i = 0; i < n; ++i) {
    int* r = &rec[9 * i];
    if (r[4] == 1) r[7] = r[8] = 0;
  }
  *count = n;
  if (records) std::memcpy(records, rec.data(), sizeof(int) * 9 * (size_t)(n < capacity ? n : capacity));
  return n <= capacity ? DA_OK : DA_ERR_WORKSPACE;
}

extern "C" int decode_max_batch(int q_len, int num_q_heads, int num_kv_heads, int head_dim, int kv_int8, int paged) {
  if (q_len < 1 || q_len > DA_MAX_QLEN || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return -DA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256) return -DA_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads * q_len > 64 || (kv_int8 && q_len != 1)) return -DA_ERR_UNSUPPORTED;
  int ng, gr, ngp, npass;
  head_groups(num_q_heads / num_kv_heads * q_len, &ng, &gr);
  group_passes(ng, head_dim, &ngp, &npass);
  return max_batch_for(head_dim, paged != 0, kv_int8 != 0, ngp);
}

// Contiguous cache, qlen query tokens per sequence (rows = Hq * qlen).
// kv8: k, v are int8 values with fp32 scales ks, vs [B, Hkv, max_ctx] (head-major).
static int contig_call(const void* q, const void* k, const void* v, const int* seq_lens, int batch, int qlen,
                int num_q_heads, int num_kv_heads, int head_dim, int max_ctx, float scale, int num_splits,
                float* part_acc, float* part_ml, unsigned long long* seg_counters, void* out, void* stream,
                bool kv8 = false, const float* ks = nullptr, const float* vs = nullptr) {
  if (qlen < 1 || qlen > DA_MAX_QLEN || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || (long long)num_q_heads * qlen > (1 << 24))
    return DA_ERR_INVALID_ARG;
  const int B = batch, Hq = num_q_heads * qlen, Hkv = num_kv_heads, D = head_dim, S = num_splits;
  if (int st = check_common(q, out, B, Hq, Hkv, D, scale, S, part_acc, part_ml, seg_counters)) return st;
  if (max_ctx < 0) return DA_ERR_INVALID_ARG;
  if (B == 0) return DA_OK;
  if (max_ctx > 0 && (!k || !v || !aligned(k, 16) || !aligned(v, 16))) return DA_ERR_INVALID_ARG;
  if (kv8 && max_ctx > 0 && (!ks || !vs || !aligned(ks, 16) || !aligned(vs, 16))) return DA_ERR_INVALID_ARG;
  if (kv8 && max_ctx % 4 != 0) return DA_ERR_UNSUPPORTED;  // scale rows are copied with 16-byte strides
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (max_ctx == 0) return zero_output(out, B, Hq, D, st);
  int dev, sms, smem_optin;
  if (current_device(&dev) || device_info(dev, &sms, &smem_optin)) return DA_ERR_CUDA;

  CUtensorMap tk, tv, tks, tvs;
  const int T = tile_tokens(D, kv8);
  if (!kv8) {
    // dims (swizzle row, token, swizzle column, head, batch): one box fills every
    // swizzle column of T tokens of one head, [D/SW][T][SW] in shared memory
    const int SW = sub_width(D);
    const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
    const cuuint64_t dims[5] = {(cuuint64_t)SW, (cuuint64_t)max_ctx, (cuuint64_t)(D / SW), (cuuint64_t)Hkv,
                                (cuuint64_t)B};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW * 2, (cuuint64_t)D * 2, row * (cuuint64_t)max_ctx};
    const cuuint32_t box[5] = {(cuuint32_t)SW, (cuuint32_t)T, (cuuint32_t)(D / SW), 1, 1};
    if (int e = encode_map(&tk, k, 5, dims, strides, box, D)) return e;
    if (int e = encode_map(&tv, v, 5, dims, strides, box, D)) return e;
  } else {
    // int8 values: dims (byte of a swizzle row, token, swizzle column, head, batch),
    // one box = [D/SW8][T][SW8] bytes of one head; scales: dims (token, head,
    // batch), one box = the T scales of one head
    const int SW8 = sub_width8(D);
    const cuuint64_t row = (cuuint64_t)Hkv * D;
    const cuuint64_t dims[5] = {(cuuint64_t)SW8, (cuuint64_t)max_ctx, (cuuint64_t)(D / SW8), (cuuint64_t)Hkv,
                                (cuuint64_t)B};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW8, (cuuint64_t)D, row * (cuuint64_t)max_ctx};
    const cuuint32_t box[5] = {(cuuint32_t)SW8, (cuuint32_t)T, (cuuint32_t)(D / SW8), 1, 1};
    const cuuint64_t sdims[3] = {(cuuint64_t)max_ctx, (cuuint64_t)Hkv, (cuuint64_t)B};
    const cuuint64_t sstrides[2] = {(cuuint64_t)max_ctx * 4, (cuuint64_t)Hkv * max_ctx * 4};
    const cuuint32_t sbox[3] = {(cuuint32_t)T, 1, 1};
    const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (int e = encode_map_t(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, swizzle8(D), k, 5, dims, strides, box)) return e;
    if (int e = encode_map_t(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, swizzle8(D), v, 5, dims, strides, box)) return e;
    if (int e = encode_map_t(&tks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, none, ks, 3, sdims, sstrides, sbox)) return e;
    if (int e = encode_map_t(&tvs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, none, vs, 3, sdims, sstrides, sbox)) return e;
  }

  Launch a;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.max_len = max_ctx;
  a.S = S;
  a.scale = scale;
  a.q = q;
  a.seq_lens = seq_lens;
  a.page_table = nullptr;
  a.page_size = 0;
  a.max_pages = 0;
  a.num_pages = 0;
  a.box_shift = 0;
  a.qlen = qlen;
  a.part_acc = part_acc;
  a.part_ml = part_ml;
  a.seg_counters = seg_counters;
  a.out = out;
  a.stream = st;
  a.paged = false;
  a.kv8 = kv8;
  a.tks = &tks;
  a.tvs = &tvs;
  return dispatch(a, tk, tv, dev, sms, smem_optin);
}

// Paged cache, qlen query tokens per sequence (rows = Hq * qlen).
// kv8: the pools hold int8 values with fp32 scale pools ks, vs [num_pages, Hkv, page_size].
static int paged_call(const void* q, const void* k_pool, const void* v_pool, const int* page_table, const int* seq_lens,
               int batch, int qlen, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
               int max_pages_per_seq, int num_pages, int max_seq_len, float scale, int num_splits, float* part_acc,
               float* part_ml, unsigned long long* seg_counters, void* out, void* stream, bool kv8 = false,
               const float* ks = nullptr, const float* vs = nullptr) {
  if (qlen < 1 || qlen > DA_MAX_QLEN || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || (long long)num_q_heads * qlen > (1 << 24))
    return DA_ERR_INVALID_ARG;
  const int B = batch, Hq = num_q_heads * qlen, Hkv = num_kv_heads, D = head_dim, S = num_splits;
  if (int st = check_common(q, out, B, Hq, Hkv, D, scale, S, part_acc, part_ml, seg_counters)) return st;
  if (page_size <= 0 || max_pages_per_seq < 0 || num_pages < 0 || max_seq_len < 0) return DA_ERR_INVALID_ARG;
  if (page_size % 16 != 0) return DA_ERR_UNSUPPORTED;
  if (B == 0) return DA_OK;
  if (!seq_lens) return DA_ERR_INVALID_ARG;
  long long cap = (long long)max_pages_per_seq * page_size;
  if (cap > max_seq_len) cap = max_seq_len;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cap == 0 || num_pages == 0) return zero_output(out, B, Hq, D, st);
  if (cap > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if (!k_pool || !v_pool || !page_table || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(page_table, 4))
    return DA_ERR_INVALID_ARG;
  if (kv8 && (!ks || !vs || !aligned(ks, 16) || !aligned(vs, 16))) return DA_ERR_INVALID_ARG;
  int dev, sms, smem_optin;
  if (current_device(&dev) || device_info(dev, &sms, &smem_optin)) return DA_ERR_CUDA;

  // One box covers R rows of one page, R = 64, 32 or 16, the largest that divides
  // the page size (tiles start on 64-token boundaries, so a box never crosses a page).
  const int box_shift = page_size % 64 == 0 ? 2 : page_size % 32 == 0 ? 1 : 0;
  const cuuint32_t R = (cuuint32_t)(16 << box_shift);
  CUtensorMap tk, tv, tks, tvs;
  if (!kv8) {
    // dims (swizzle row, row in page, swizzle column, head, page): one box fills every
    // swizzle column of its rows, [D/SW][R][SW] in shared memory
    const int SW = sub_width(D);
    const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
    const cuuint64_t dims[5] = {(cuuint64_t)SW, (cuuint64_t)page_size, (cuuint64_t)(D / SW), (cuuint64_t)Hkv,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW * 2, (cuuint64_t)D * 2, row * (cuuint64_t)page_size};
    const cuuint32_t box[5] = {(cuuint32_t)SW, R, (cuuint32_t)(D / SW), 1, 1};
    if (int e = encode_map(&tk, k_pool, 5, dims, strides, box, D)) return e;
    if (int e = encode_map(&tv, v_pool, 5, dims, strides, box, D)) return e;
  } else {
    // int8 values: dims (byte of a swizzle row, row in page, swizzle column, head,
    // page), one box = [D/SW8][R][SW8] bytes; scales: dims (row in page, head,
    // page), one box = R scales of one head
    const int SW8 = sub_width8(D);
    const cuuint64_t row = (cuuint64_t)Hkv * D;
    const cuuint64_t dims[5] = {(cuuint64_t)SW8, (cuuint64_t)page_size, (cuuint64_t)(D / SW8), (cuuint64_t)Hkv,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[4] = {row, (cuuint64_t)SW8, (cuuint64_t)D, row * (cuuint64_t)page_size};
    const cuuint32_t box[5] = {(cuuint32_t)SW8, R, (cuuint32_t)(D / SW8), 1, 1};
    const cuuint64_t sdims[3] = {(cuuint64_t)page_size, (cuuint64_t)Hkv, (cuuint64_t)num_pages};
    const cuuint64_t sstrides[2] = {(cuuint64_t)page_size * 4, (cuuint64_t)Hkv * page_size * 4};
    const cuuint32_t sbox[3] = {R, 1, 1};
    const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (int e = encode_map_t(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, swizzle8(D), k_pool, 5, dims, strides, box)) return e;
    if (int e = encode_map_t(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, swizzle8(D), v_pool, 5, dims, strides, box)) return e;
    if (int e = encode_map_t(&tks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, none, ks, 3, sdims, sstrides, sbox)) return e;
    if (int e = encode_map_t(&tvs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, none, vs, 3, sdims, sstrides, sbox)) return e;
  }

  Launch a;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.max_len = (int)cap;
  a.S = S;
  a.scale = scale;
  a.q = q;
  a.seq_lens = seq_lens;
  a.page_table = page_table;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.box_shift = box_shift;
  a.qlen = qlen;
  a.part_acc = part_acc;
  a.part_ml = part_ml;
  a.seg_counters = seg_counters;
  a.out = out;
  a.stream = st;
  a.paged = true;
  a.kv8 = kv8;
  a.tks = &tks;
  a.tvs = &tvs;
  return dispatch(a, tk, tv, dev, sms, smem_optin);
}

extern "C" int decode_attn_contig(const void* q, const void* k, const void* v, const int* seq_lens, int batch,
                                  int num_q_heads, int num_kv_heads, int head_dim, int max_ctx, float scale,
                                  int num_splits, float* part_acc, float* part_ml,
                                  unsigned long long* seg_counters, void* out, void* stream) {
  return contig_call(q, k, v, seq_lens, batch, 1, num_q_heads, num_kv_heads, head_dim, max_ctx, scale, num_splits,
                     part_acc, part_ml, seg_counters, out, stream);
}

extern "C" int decode_attn_paged(const void* q, const void* k_pool, const void* v_pool, const int* page_table,
                                 const int* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int page_size, int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                                 int num_splits, float* part_acc, float* part_ml, unsigned long long* seg_counters,
                                 void* out, void* stream) {
  return paged_call(q, k_pool, v_pool, page_table, seq_lens, batch, 1, num_q_heads, num_kv_heads, head_dim,
                    page_size, max_pages_per_seq, num_pages, max_seq_len, scale, num_splits, part_acc, part_ml,
                    seg_counters, out, stream);
}

extern "C" int decode_attn_multi_contig(const void* q, const void* k, const void* v, const int* seq_lens, int batch,
                                        int q_len, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx,
                                        float scale, int num_splits, float* part_acc, float* part_ml,
                                        unsigned long long* seg_counters, void* out, void* stream) {
  return contig_call(q, k, v, seq_lens, batch, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx, scale,
                     num_splits, part_acc, part_ml, seg_counters, out, stream);
}

extern "C" int decode_attn_multi_paged(const void* q, const void* k_pool, const void* v_pool, const int* page_table,
                                       const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads,
                                       int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                                       int max_seq_len, float scale, int num_splits, float* part_acc, float* part_ml,
                                       unsigned long long* seg_counters, void* out, void* stream) {
  return paged_call(q, k_pool, v_pool, page_table, seq_lens, batch, q_len, num_q_heads, num_kv_heads, head_dim,
                    page_size, max_pages_per_seq, num_pages, max_seq_len, scale, num_splits, part_acc, part_ml,
                    seg_counters, out, stream);
}

extern "C" int decode_attn_int8_contig(const void* q, const void* k_i8, const void* v_i8, const float* k_scale,
                                       const float* v_scale, const int* seq_lens, int batch, int num_q_heads,
                                       int num_kv_heads, int head_dim, int max_ctx, float scale, int num_splits,
                                       float* part_acc, float* part_ml, unsigned long long* seg_counters, void* out,
                                       void* stream) {
  return contig_call(q, k_i8, v_i8, seq_lens, batch, 1, num_q_heads, num_kv_heads, head_dim, max_ctx, scale,
                     num_splits, part_acc, part_ml, seg_counters, out, stream, true, k_scale, v_scale);
}

extern "C" int decode_attn_int8_paged(const void* q, const void* k_pool_i8, const void* v_pool_i8,
                                      const float* k_scale_pool, const float* v_scale_pool, const int* page_table,
                                      const int* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                      int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                                      float scale, int num_splits, float* part_acc, float* part_ml,
                                      unsigned long long* seg_counters, void* out, void* stream) {
  return paged_call(q, k_pool_i8, v_pool_i8, page_table, seq_lens, batch, 1, num_q_heads, num_kv_heads, head_dim,
                    page_size, max_pages_per_seq, num_pages, max_seq_len, scale, num_splits, part_acc, part_ml,
                    seg_counters, out, stream, true, k_scale_pool, v_scale_pool);
}

extern "C" int decode_combine(const float* part_acc, const float* part_ml, int batch, int num_q_heads,
                              int head_dim, int num_splits, void* out, void* stream) {
  const int B = batch, Hq = num_q_heads, D = head_dim, S = num_splits;
  if (B < 0 || Hq <= 0 || S < 1 || S > DA_MAX_SPLITS) return DA_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128 && D != 256) return DA_ERR_UNSUPPORTED;
  if (B == 0) return DA_OK;
  if (!part_acc || !part_ml || !out) return DA_ERR_INVALID_ARG;
  if (!aligned(part_acc, 16) || !aligned(part_ml, 8) || !aligned(out, 16)) return DA_ERR_INVALID_ARG;
  int dev, sms, smem_optin;
  if (current_device(&dev) || device_info(dev, &sms, &smem_optin)) return DA_ERR_CUDA;
  CombineParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.part_acc = part_acc;
  cp.part_ml = part_ml;
  cp.out = reinterpret_cast<__nv_bfloat16*>(out);
  cp.B = B;
  cp.Hq = Hq;
  cp.S = S;
  cp.planned = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (D) {
    case 32: return launch_combine<32>(cp, dev, sms, st, false);
    case 64: return launch_combine<64>(cp, dev, sms, st, false);
    case 128: return launch_combine<128>(cp, dev, sms, st, false);
    default: return launch_combine<256>(cp, dev, sms, st, false);
  }
}

extern "C" const char* decode_status_string(int status) {
  switch (status) {
    case DA_OK: return "DA_OK";
    case DA_ERR_INVALID_ARG: return "DA_ERR_INVALID_ARG";
    case DA_ERR_UNSUPPORTED: return "DA_ERR_UNSUPPORTED";
    case DA_ERR_WORKSPACE: return "DA_ERR_WORKSPACE";
    case DA_ERR_CUDA: return "DA_ERR_CUDA";
    case DA_ERR_TIMEOUT: return "DA_ERR_TIMEOUT";
    default: return "unknown status";
  }
}

// One CTA waits on an mbarrier that expects an arrival nobody makes; the bounded
// wait gives up after the timeout and records it in the device error word.
__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, &abort_flag, timeout_ns);
  __syncthreads();
}

extern "C" int decode_selftest_bounded_wait(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return DA_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(timeout_ns);
  if (cudaGetLastError() != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

extern "C" int decode_device_error(void* stream, unsigned int* flags) {
  if (!flags) return DA_ERR_INVALID_ARG;
  *flags = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  unsigned int w = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess) {
    cudaGetLastError();
    return DA_ERR_CUDA;
  }
  if (w) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return DA_ERR_CUDA;
    }
  }
  *flags = w;
  return w ? DA_ERR_TIMEOUT : DA_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of decode_attn_contig.
//
// Some callers cannot hand this library any device workspace: a runtime that
// owns a fixed device-memory budget and passes its plugins nothing but input
// and output buffers, or a serving loop that must not call cudaMalloc (which
// can synchronise the device) between steps.  For them the segment counters and
// the split partials live in the file-scope array below instead of caller
// buffers.  Every GPU that loads this library holds the array (8 MiB) until the
// process exits.
//
// Host code may not use the array's name as a device address (on the host it
// names a shadow variable), so its device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, by the first call on it.
// All calls share the array: two calls that overlap on the GPU (different
// streams or threads) race on it.
//
// Layout: the segment counters come first, at a fixed offset, with room for
// kNoAllocMaxSegments of them, so counter words only ever hold counter values
// (epoch << 32 | state), whatever shapes earlier calls had; the array starts
// zeroed, and a stale counter from another call counts as zero.  The partials
// follow; every partial slot a merge reads is written earlier in the same call,
// so they need no clearing.
// ---------------------------------------------------------------------------

namespace da {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
constexpr size_t kNoAllocMaxSegments = 16384;  // 128 KB of counters
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kMaxDevices] = {nullptr};
}  // namespace
}  // namespace da

static __device__ __align__(256) unsigned char g_noalloc_scratch[da::kNoAllocScratchBytes];

extern "C" int decode_attn_contig_noalloc(const void* q, const void* k, const void* v, const int* seq_lens,
                                          int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_ctx, float scale, void* out, void* stream) {
  const int B = batch, Hq = num_q_heads, Hkv = num_kv_heads, D = head_dim;
  if (max_ctx < 0) return DA_ERR_INVALID_ARG;
  // the argument checks of decode_attn_contig come first, so a bad argument gets
  // the same status from both entry points
  if (int st = check_common(q, out, B, Hq, Hkv, D, scale, 1, nullptr, nullptr, nullptr)) return st;
  if (B == 0) return DA_OK;
  int dev, sms, smem_optin;
  if (current_device(&dev) || device_info(dev, &sms, &smem_optin)) return DA_ERR_CUDA;
  const int S = decode_num_splits(B, Hkv, max_ctx, D, sms);
  if (S < 1) return DA_ERR_INVALID_ARG;
  float* acc = nullptr;
  float* ml = nullptr;
  unsigned long long* ctr = nullptr;
  if (S >= 2) {
    const size_t segments = (size_t)B * Hkv * ((Hq / Hkv + 7) / 8);  // at least B * U
    const size_t ctr_bytes = kNoAllocMaxSegments * 8;
    const size_t acc_bytes = ((size_t)B * Hq * S * D * 4 + 255) / 256 * 256;
    const size_t ml_bytes = (size_t)B * Hq * S * 2 * 4;
    if (segments > kNoAllocMaxSegments || ctr_bytes + acc_bytes + ml_bytes > kNoAllocScratchBytes)
      return DA_ERR_WORKSPACE;
    unsigned char* base = nullptr;
    {
      std::lock_guard<std::mutex> lk(g_noalloc_mu);
      if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
          cudaGetLastError();
          return DA_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
      }
      base = g_noalloc_ptr[dev];
    }
    ctr = reinterpret_cast<unsigned long long*>(base);
    acc = reinterpret_cast<float*>(base + ctr_bytes);
    ml = reinterpret_cast<float*>(base + ctr_bytes + acc_bytes);
  }
  return decode_attn_contig(q, k, v, seq_lens, B, Hq, Hkv, D, max_ctx, scale, S, acc, ml, ctr, out, stream);
}

// ------------------------------------------------------------------ prefill
// The causal prefill entry points (prefill_attn_contig / prefill_attn_paged) are
// in prefill_host.cuh, kept apart so that the decode and prefill sources can be
// told apart (the measurement scripts tie ncu figures to the sources they came from).
#include "prefill_host.cuh"
