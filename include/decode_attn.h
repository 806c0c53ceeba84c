/*
 * decode_attn.h — C ABI of the split-KV GQA decode-attention library (GB300, sm_103a).
 *
 * One query token per sequence attends over that sequence's bf16 KV cache.  For
 * sequence b, query head h and KV head g = h / G (G = Hq / Hkv; the G query heads
 * of a KV head are consecutive), over the L_b cached tokens t:
 *
 *     s_t = scale * <q[b,h,:], k[b,t,g,:]>,   out[b,h,:] = sum_t softmax(s)_t * v[b,t,g,:]
 *
 * in fp32 on the GPU, rounded once to bf16.  The G query heads of a KV head share
 * every K/V tile they read (head packing, AstrAI commit 988e013 "csrc", MMA decode
 * items).  The token range of each (sequence, KV head) is cut into pieces processed
 * by different CTAs; each piece leaves unnormalised partials (acc, m, l) and a
 * log-sum-exp combine merges them (AstrAI commit 988e013, split-KV items; merge
 * order as in "perf(qwen3.8): split the flash-decode KV range across warp-groups",
 * section "Mechanism").  Paged caches are read through a page table (AstrAI commit
 * 69fecaf "csrc/tests", paged decode items).
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates nothing, keeps no per-call state, never synchronises the stream and
 *    enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    of the current device.
 *  - bf16 tensors are passed as `void*` (__nv_bfloat16 elements); fp32 as float*.
 *  - q, k, v, k_pool, v_pool, out must be 16-byte aligned; part_acc and part_ml
 *    16-byte and 8-byte aligned.
 *  - Every argument is checked on the host first; a bad argument returns
 *    DA_ERR_INVALID_ARG or DA_ERR_UNSUPPORTED and launches nothing.  A launch
 *    failure returns DA_ERR_CUDA (the CUDA error is cleared).
 *  - Supported: head_dim in {32, 64, 128, 256}; Hq % Hkv == 0; 1 <= G <= 64;
 *    1 <= num_splits <= DA_MAX_SPLITS; page_size a multiple of 16.
 *  - Device waits are bounded: a kernel that waits too long sets a device error
 *    word and returns; decode_device_error() reads it.
 *
 * The split plan.  Work is counted in 16-token blocks, n_b = ceil(L_b / 16).
 * The query heads of one KV head form ceil(G / 8) equal sub-groups of at most 8
 * rows; one pass over the KV head runs ngp of them (the largest power of two that
 * divides their number, at most 2 for head_dim 128 and 4 otherwise), so a
 * sequence has U = Hkv * ceil(G / 8) / ngp segment slots (U = Hkv when G <= 8).
 * The segments (b, u) lie end to end on one line in (u, b) order (slot-major);
 * segment (b, u) takes w_b = c + 4*ceil(n_b / 4) positions, c = 4*ceil((2816 /
 * head_dim) / 4) of them without blocks (they stand for the fixed cost of a
 * piece), then its n_b blocks, then padding to whole 64-token units; an empty
 * sequence takes none.  P_b = w_0 + ... + w_{b-1}; segment (b, u) starts at
 * u*P_B + P_b; NB = U * P_B positions in all.
 *   num_splits == 1: every segment is computed whole and written directly.
 *   num_splits >= 2: the line is cut into ranges of q positions, q = ceil(NB / R)
 *     with R = (num_splits - 1) * U, rounded up to a multiple of 4 (at least 4);
 *     each range is one CTA's work; the pieces of a segment are the non-empty sets
 *     of its blocks that share a range (index j = r - range of its first block),
 *     at most num_splits of them.  A segment with one piece is written directly;
 *     one with several leaves partials in slots j = 0..pieces-1, which are merged
 *     into the output by the CTA that finishes its last piece (found with the
 *     segment's counter) when there are at most 8, else by a combine kernel that
 *     follows as a programmatic dependent launch (one CTA alone would need several
 *     dependent rounds of L2 reads for a long run of partials); an empty sequence
 *     (L_b == 0) gets a zero output.
 *   decode_plan_pieces reports this partition, and what every partial slot holds
 *   when a call returns, for any shape (host only).
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DA_OK = 0,
  DA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, Hq % Hkv != 0, ... */
  DA_ERR_UNSUPPORTED = 2,  /* head_dim, page_size, group size or batch outside the built kernels */
  DA_ERR_WORKSPACE = 3,    /* num_splits >= 2 but part_acc / part_ml / seg_counters missing */
  DA_ERR_CUDA = 4,         /* a CUDA call or launch failed (error cleared) */
  DA_ERR_TIMEOUT = 5       /* a kernel gave up on a bounded wait (see decode_device_error) */
} da_status;

#define DA_MAX_SPLITS 1024
#define DA_MAX_QLEN 16  /* query tokens per sequence of decode_attn_multi_* */

/*
 * decode_num_splits — the split count for a decode shape (host only, pure).
 *
 * The pages choose a split count that fills the device, capped by the tile count
 * (AstrAI commit 988e013, split-KV items; AstrAI commit 69fecaf, planner items).
 * Here it is the number of partial slots that lets every CTA of the persistent
 * grid own one range: S = ceil(C / num_kv_heads) + 1 with C = num_sms (one CTA per
 * SM), capped by ceil(max_seq_len / 16) and DA_MAX_SPLITS; S = 1 when
 * max_seq_len <= 16.  batch is accepted for interface stability and does not
 * change the result.  num_sms <= 0 queries the current device.
 * Returns S >= 1, or -DA_ERR_INVALID_ARG / -DA_ERR_CUDA.
 */
int decode_num_splits(int batch, int num_kv_heads, int max_seq_len, int head_dim, int num_sms);

/*
 * decode_attn_contig — decode attention over a contiguous cache.
 *
 *  q        bf16 [batch, num_q_heads, head_dim]
 *  k, v     bf16 [batch, max_ctx, num_kv_heads, head_dim]  (token-major rows)
 *  seq_lens int32 [batch] on the device, or NULL (every sequence has max_ctx tokens);
 *           values are clamped to [0, max_ctx]
 *  scale    finite float multiplying q.k (applied in fp32 after the dot product)
 *  num_splits, part_acc float [batch, num_q_heads, num_splits, head_dim],
 *           part_ml float [batch, num_q_heads, num_splits, 2] = (m, l) with m in
 *           natural-log units of the scaled score: caller-owned scratch, unused
 *           (may be NULL) when num_splits == 1.  Slots the plan does not use are not
 *           written.
 *  seg_counters  uint64 [batch * num_kv_heads * ceil(G / 8)] (at least batch * U entries are
 *           used): caller-owned, zeroed once before the first call and then
 *           reusable by every later call (each call tags its updates with its own
 *           epoch, and a value left by another call counts as zero, so no reset is
 *           needed, even after a failed call); unused (may be NULL) when
 *           num_splits == 1.  Calls that share partial buffers or counters must
 *           not overlap on the GPU.  A call may be captured in a CUDA graph and
 *           replayed: a completed call leaves each counter it used holding a value
 *           that every later call, replays included, counts as zero.  Only after a
 *           call that ended in DA_ERR_TIMEOUT must the counters be zeroed again
 *           before a captured graph that uses them is replayed.
 *  Batch limit: the split kernel keeps 8 bytes of plan per sequence in shared
 *           memory, so batch is at most decode_max_batch(...) for the shape
 *           (1159 for bf16 head_dim 128 with G <= 8); a larger batch returns
 *           DA_ERR_UNSUPPORTED and launches nothing.
 *  out      bf16 [batch, num_q_heads, head_dim]
 *  stream   cudaStream_t
 * Enqueues the split kernel, and the combine kernel when num_splits > 8.
 */
int decode_attn_contig(const void* q, const void* k, const void* v, const int* seq_lens,
                       int batch, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx,
                       float scale, int num_splits, float* part_acc, float* part_ml,
                       unsigned long long* seg_counters, void* out, void* stream);

/*
 * decode_attn_paged — decode attention over a paged cache.
 *
 *  k_pool, v_pool bf16 [num_pages, page_size, num_kv_heads, head_dim]
 *  page_table     int32 [batch, max_pages_per_seq] on the device: token t of
 *                 sequence b is row t % page_size of page page_table[b, t / page_size].
 *                 Entries past ceil(L_b / page_size) are never read.  Entries that
 *                 are read must lie in [0, num_pages); one that does not sets bit 2
 *                 of the device error word (decode_device_error) and reads page 0.
 *  seq_lens       int32 [batch] on the device (required); clamped to
 *                 [0, min(max_seq_len, max_pages_per_seq * page_size)]
 *  Other arguments as for decode_attn_contig.  Each 16-token block is fetched from
 *  its page with one tile copy, so page_size must be a multiple of 16.
 */
int decode_attn_paged(const void* q, const void* k_pool, const void* v_pool,
                      const int* page_table, const int* seq_lens,
                      int batch, int num_q_heads, int num_kv_heads, int head_dim,
                      int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                      float scale, int num_splits, float* part_acc, float* part_ml,
                      unsigned long long* seg_counters, void* out, void* stream);

/*
 * decode_combine — stand-alone log-sum-exp merge of split partials.
 *
 * For each (b, h): M = max over slots j < num_splits with l_j > 0 of m_j,
 * w_j = exp(m_j - M), out = sum_j w_j acc_j / sum_j w_j l_j, summed in a fixed
 * order (bitwise reproducible); slots with l_j == 0 are skipped and a row with no
 * live slot is written as zeros
 * ("perf(qwen3.8): split the flash-decode KV range across warp-groups", section
 * "Mechanism"; AstrAI commit 988e013, combine kernel).  Every slot is read, so
 * unused slots must hold l == 0.  Layouts as in decode_attn_contig.
 */
int decode_combine(const float* part_acc, const float* part_ml, int batch, int num_q_heads,
                   int head_dim, int num_splits, void* out, void* stream);

/*
 * decode_attn_contig_noalloc — decode_attn_contig for callers that cannot allocate.
 *
 * For callers that may not allocate device memory or hold any workspace of
 * their own: a runtime with a fixed device-memory budget that hands its plugins
 * only input and output buffers, or a serving loop that must not call cudaMalloc
 * (which can synchronise the device) between steps.  The source pages have no
 * such entry point; it is specific to this library.  Arguments are those of
 * decode_attn_contig without num_splits, part_acc, part_ml and seg_counters: the
 * split count is decode_num_splits(batch, num_kv_heads, max_ctx, head_dim, <SMs of
 * the device>), and the segment counters and partials live in an 8 MiB array
 * inside the library (every GPU that loads the library holds it until exit).
 * The array holds at most 16384 segments (batch * num_kv_heads * ceil(G / 8)) and
 * batch * num_q_heads * S * head_dim * 4 bytes of partial values (rounded up to
 * 256) plus batch * num_q_heads * S * 8 bytes of (m, l) in 8 MiB - 128 KiB;
 * larger shapes return DA_ERR_WORKSPACE and launch nothing.  Argument errors
 * return the status decode_attn_contig returns for them.  The first call on a
 * device looks up the array's device address (no allocation); make that first
 * call before any stream capture.  Calls share the array: calls that overlap on
 * the GPU race.  Calls no cudaMalloc, cudaFree or allocating library routine.
 */
int decode_attn_contig_noalloc(const void* q, const void* k, const void* v, const int* seq_lens,
                               int batch, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx,
                               float scale, void* out, void* stream);

/*
 * decode_num_splits_multi — the split count for a shape given its query heads and
 * query tokens per sequence (host only, pure): decode_num_splits with the KV
 * heads counted once per pass.  The G * q_len rows of a KV head form ceil(G*q_len/8)
 * sub-groups of at most 8 rows; one pass over the KV head runs ngp of them, the
 * largest power of two that divides their number, at most 2 for head_dim 128 and
 * 4 otherwise; so a sequence has num_kv_heads * (sub-groups / ngp) segments.
 * Gives the same value as decode_num_splits when G * q_len <= 8.  Returns
 * -DA_ERR_INVALID_ARG / -DA_ERR_UNSUPPORTED for bad shapes.
 */
int decode_num_splits_multi(int batch, int q_len, int num_q_heads, int num_kv_heads, int max_seq_len,
                            int head_dim, int num_sms);

/*
 * decode_plan_pieces — the partition of a decode call into pieces (host only, pure).
 *
 * Reports, for a call with these sizes, host copies of its sequence lengths and
 * num_splits, every piece the split kernel computes: the same plan code runs
 * here on the host.  The pages fix only caps on the split count (AstrAI commit
 * 988e013 "csrc", split-KV items: at most the tile count and 32 splits); the
 * partition itself is this library's (see "The split plan" above), and any
 * partition of each segment into at most num_splits pieces gives the same
 * attention output.
 *  seq_lens   int32 [batch] on the HOST, or NULL (every sequence max_len tokens);
 *             clamped to [0, max_len]
 *  q_len      query tokens per sequence (1 for decode_attn_contig / _paged);
 *             rows of a sequence are num_q_heads * q_len (head-major)
 *  max_len    the call's length cap: max_ctx (contiguous) or
 *             min(max_pages_per_seq * page_size, max_seq_len) (paged)
 *  records    int32 [capacity][9], one record per piece in CTA walk order:
 *             (b, row0, nrows, j, npieces, t0, t1, held_t0, held_t1): sequence b,
 *             rows row0 .. row0 + nrows - 1 of the pass (query heads x q_len
 *             rows, head-major), partial slot j of npieces, tokens [t0, t1), and
 *             the token range whose partial slot j holds when the call returns
 *             ([t0, t1); held_t0 == held_t1 == 0 when the segment has one piece,
 *             which is written straight to the output).  Empty sequences
 *             have no pieces.
 * *count receives the number of pieces; at most capacity records are written.
 * Returns DA_OK, DA_ERR_WORKSPACE (capacity < *count; *count is still set),
 * DA_ERR_INVALID_ARG or DA_ERR_UNSUPPORTED.
 */
int decode_plan_pieces(const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_len, int num_splits, int* records, int capacity, int* count);

/*
 * decode_max_batch — the largest batch the decode kernels accept for a shape
 * (host only, pure): the split kernel keeps two ints of plan per sequence in
 * shared memory beside its K/V stages.  q_len and the heads are as for
 * decode_num_splits_multi; kv_int8 != 0 for the int8 cache entry points, paged
 * != 0 for paged caches.  Returns the limit, or -DA_ERR_INVALID_ARG /
 * -DA_ERR_UNSUPPORTED.
 */
int decode_max_batch(int q_len, int num_q_heads, int num_kv_heads, int head_dim, int kv_int8, int paged);

/*
 * decode_attn_multi_contig / decode_attn_multi_paged — multi-query decode, the
 * verification step of speculative decoding scored on "perf(dspark): overlap KV
 * staging with compute via cp.async", section "sparkinfer DSpark auto-eval —
 * eval-dspark:XL" (a draft block of 7): every sequence scores q_len new tokens at once, the last q_len of its
 * L_b cached tokens, causally within the block.  Query token i (0-based) of
 * sequence b attends to cached tokens [0, L_b - q_len + 1 + i); a token that
 * sees none (L_b < q_len - i) gets a zero output.  q_len == 1 is exactly
 * decode_attn_contig / decode_attn_paged.
 *  q, out        bf16 [batch, num_q_heads, q_len, head_dim] (head-major: the q_len
 *                rows of one head are consecutive)
 *  part_acc      float [batch, num_q_heads, q_len, num_splits, head_dim];
 *  part_ml       float [batch, num_q_heads, q_len, num_splits, 2]
 *  seg_counters  uint64 [batch * num_kv_heads * ceil(G * q_len / 8)], zeroed once
 *  Every other argument as for decode_attn_contig / decode_attn_paged (the same
 *  split plan, with G * q_len rows per KV head in sub-groups of at most 8).
 *  1 <= q_len <= DA_MAX_QLEN and G * q_len <= 64, else DA_ERR_INVALID_ARG /
 *  DA_ERR_UNSUPPORTED.  num_splits: decode_num_splits_multi(batch, q_len, ...).
 */
int decode_attn_multi_contig(const void* q, const void* k, const void* v, const int* seq_lens, int batch,
                             int q_len, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx, float scale,
                             int num_splits, float* part_acc, float* part_ml, unsigned long long* seg_counters,
                             void* out, void* stream);
int decode_attn_multi_paged(const void* q, const void* k_pool, const void* v_pool, const int* page_table,
                            const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                            float scale, int num_splits, float* part_acc, float* part_ml,
                            unsigned long long* seg_counters, void* out, void* stream);

/*
 * decode_attn_int8_contig / decode_attn_int8_paged — decode over an int8 KV cache.
 * "perf(dspark): overlap KV staging with compute via cp.async", section "Cost and
 * fallbacks", names an int8 pool read through a dequant-into-shared-memory path; its
 * format is not given there.  Here K and V are symmetric int8 values with one fp32
 * scale per (token, KV head): K[t, g, :] = k_i8[t, g, :] * k_scale[g, t] (V likewise).
 *  k_i8, v_i8       int8 [batch, max_ctx, num_kv_heads, head_dim] (16-byte aligned)
 *  k_scale, v_scale float [batch, num_kv_heads, max_ctx], head-major (16-byte aligned;
 *                   max_ctx a multiple of 4)
 *  paged:  k_pool_i8, v_pool_i8 int8 [num_pages, page_size, num_kv_heads, head_dim],
 *          k_scale_pool, v_scale_pool float [num_pages, num_kv_heads, page_size]
 *  Every other argument, the split plan, the partials and the error behaviour are
 *  those of decode_attn_contig / decode_attn_paged.  The MMA warps widen the int8
 *  operands of each 16-token block to f16 in registers (exact) and multiply in f16
 *  with fp32 accumulation; K's scale multiplies a token's score and V's scale its
 *  probability.  q is converted to f16, exact for |q| in [2^-14, 65504].
 */
int decode_attn_int8_contig(const void* q, const void* k_i8, const void* v_i8, const float* k_scale,
                            const float* v_scale, const int* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                            int head_dim, int max_ctx, float scale, int num_splits, float* part_acc, float* part_ml,
                            unsigned long long* seg_counters, void* out, void* stream);
int decode_attn_int8_paged(const void* q, const void* k_pool_i8, const void* v_pool_i8, const float* k_scale_pool,
                           const float* v_scale_pool, const int* page_table, const int* seq_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size, int max_pages_per_seq,
                           int num_pages, int max_seq_len, float scale, int num_splits, float* part_acc,
                           float* part_ml, unsigned long long* seg_counters, void* out, void* stream);

/*
 * prefill_attn_contig / prefill_attn_paged — causal GQA attention of a chunk of
 * q_len new tokens per sequence (prefill when the chunk is the whole sequence,
 * chunked prefill otherwise).  "gqa_prefill_attn" on the AstrAI commit page
 * ("csrc", commit 988e013) is a tiled shared-memory kernel with mask support; the
 * pages fix no layout, so: sequence b holds L_b cached tokens (its chunk included,
 * already written to the cache), the chunk is its last q_len tokens, and query
 * token i (position L_b - q_len + i) attends to positions 0 .. L_b - q_len + i.  A
 * query that sees no token (L_b < q_len - i) gives zeros.  Query head h reads KV
 * head h / G.
 *  q, out   bf16 [batch, q_len, num_q_heads, head_dim], token-major (16-byte aligned)
 *  k, v     the decode cache: contiguous [batch, max_ctx, num_kv_heads, head_dim]
 *           (seq_lens may be NULL: every sequence max_ctx tokens), or pools
 *           [num_pages, page_size, num_kv_heads, head_dim] with page_table
 *           int32 [batch, max_pages_per_seq] (page_size a multiple of 16)
 *  seq_lens int32 [batch], clamped to [0, max_ctx] (paged: to
 *           min(max_pages_per_seq * page_size, max_seq_len))
 *  head_dim 32, 64, 128 or 256; G = num_q_heads / num_kv_heads <= 64.
 *  scale    any finite value (a positive one is applied in the exponent's fma).
 * Softmax in fp32 (log2 units), P rounded to bf16 for the P V product, fp32
 * accumulation, output rounded to bf16.  head_dim 64, 128 and 256 run on the
 * tcgen05 tensor cores with the S and O accumulators in tensor memory; head_dim
 * 32 on warp-level MMAs.  No workspace; the library allocates nothing.  Argument
 * errors return DA_ERR_INVALID_ARG / DA_ERR_UNSUPPORTED before any launch; so
 * does a build whose tensor-core kernel was compiled with fewer registers per
 * thread than its warpgroup split needs (DA_ERR_UNSUPPORTED).  Page-table entries
 * outside [0, num_pages) set bit 2 of the device error word (decode_device_error)
 * and read page 0 instead.
 */
int prefill_attn_contig(const void* q, const void* k, const void* v, const int* seq_lens, int batch, int q_len,
                        int num_q_heads, int num_kv_heads, int head_dim, int max_ctx, float scale, void* out,
                        void* stream);
int prefill_attn_paged(const void* q, const void* k_pool, const void* v_pool, const int* page_table,
                       const int* seq_lens, int batch, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int page_size, int max_pages_per_seq, int num_pages, int max_seq_len, float scale, void* out,
                       void* stream);

/* Human-readable name of a da_status value (static string). */
const char* decode_status_string(int status);

/*
 * decode_device_error — synchronise `stream`, then read and clear the device error
 * word of the current device.  *flags receives the word: bit 0 a kernel gave up on
 * a bounded wait, bit 1 a segment-counter update gave up, bit 2 a page-table entry
 * read by decode_attn_paged / decode_attn_multi_paged / decode_attn_int8_paged was
 * outside [0, num_pages)
 * (that box was read from page 0 instead, so the affected rows are wrong but no
 * copy leaves the pool).  Returns DA_OK when flags == 0, DA_ERR_TIMEOUT otherwise,
 * or DA_ERR_CUDA.
 */
int decode_device_error(void* stream, unsigned int* flags);

/*
 * decode_selftest_bounded_wait — diagnostic of the bounded waits that every
 * kernel of this library uses (the pages have no counterpart).  Enqueues on
 * `stream` one CTA that waits on a shared-memory mbarrier that nothing ever
 * completes; the wait gives up after timeout_ns nanoseconds of the GPU's global
 * timer, sets bit 0 of the device error word and the kernel returns normally, so
 * the context stays usable.  decode_device_error() then reports DA_ERR_TIMEOUT
 * with flags bit 0 set.  timeout_ns must be in (0, 10^9]; returns DA_OK,
 * DA_ERR_INVALID_ARG or DA_ERR_CUDA (launch failure).
 */
int decode_selftest_bounded_wait(unsigned long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
