/*
 * mj.h — C ABI of libmj: paged decode attention over an e4m3 or packed e2m3 (e3m2, e2m1)
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * One decode step is four calls, in the order the mjolnir-kernel README
 * lists them ("A decode step", items 1-4):
 *
 *   mj_plan_split_kv    (host)   split-KV work list sized to one wave of CTAs
 *   mj_quantize_q       (device) dynamic per-(request, KV head) e4m3 Q
 *   mj_decode_attention (device) stream KV pages through the block table,
 *                                online softmax, P.V
 *   mj_merge_lse        (device) merge split-KV partials by log-sum-exp
 *
 * and, before the step, the cache write of the new tokens:
 *
 *   mj_write_kv         (device) quantize K/V rows into the paged caches
 *
 * Conventions (all calls):
 *  - Every call returns an mj_status; 0 is success, negative is an error.
 *    Nothing throws, aborts or prints.
 *  - No call allocates device or host memory and no call synchronises the
 *    device. All memory is the caller's: device tensors, the plan staging
 *    buffers, and a device workspace of mj_workspace_size() bytes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *    Device calls only enqueue work on it; argument errors are detected on
 *    the host before anything is enqueued.
 *  - Device pointers must be 16-byte aligned (the runner page's _ptr
 *    rejects other base pointers); packed
 *    (e2m3, e3m2, e2m1) K/V bases must be 32-byte aligned (T5DecodeRunner._kv_ptr).
 *  - Q and O strides are in ELEMENTS; K/V strides are in BYTES, so e4m3 and
 *    packed e2m3 caches share one convention.
 *  - Launch shapes depend only on the arguments (the grid is the plan's
 *    padded num_work), never on device data, so a step can be captured in a
 *    CUDA graph and replayed with new plans written into the same buffers
 *    (runner page, module docstring: the plan's buffers keep their
 *    addresses and the grid keeps its size per q_len, so a captured graph
 *    stays valid). The first launch of a kernel configuration on a device
 *    raises its shared-memory limit and queries its occupancy (host calls,
 *    cached): make one call of each configuration before capturing it.
 */
#ifndef MJ_H
#define MJ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MJ_API __attribute__((visibility("default")))
#else
#define MJ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mj_status {
  MJ_OK = 0,
  MJ_ERR_INVALID_ARG = -1,  /* null pointer, negative or inconsistent size */
  MJ_ERR_UNSUPPORTED = -2,  /* valid but not implemented (head size, page size, format) */
  MJ_ERR_ALIGNMENT = -3,    /* pointer or stride alignment rule broken */
  MJ_ERR_CAPACITY = -4,     /* a caller buffer (pad_to, workspace) is too small */
  MJ_ERR_CUDA = -5,         /* a CUDA runtime call failed (launch, symbol lookup) */
  MJ_ERR_DEVICE_CHECK = -6  /* a kernel recorded an anomaly in the workspace status word */
} mj_status;

/* KV cache formats. The narrow ones (e2m3, e3m2, e2m1; OCP FP6 / FP4, no NaN)
 * take per-(KV head, channel) scales folded into q_mul / o_mul, fp8 Q only,
 * and 32-byte aligned cache bases. The package README lists e3m2 and e2m1
 * beside e2m3 ("Beyond fp8: the harness"); their packing is this library's
 * reading: e3m2 as e2m3, e2m1 two codes per byte, low nibble first. */
typedef enum mj_kv_format {
  MJ_KV_E4M3 = 0,  /* one e4m3 code per byte; row = d bytes */
  MJ_KV_E2M3 = 1,  /* packed e2m3: 4 codes per 3 bytes, little-endian bitstream; row = d*3/4 bytes */
  MJ_KV_E3M2 = 2,  /* packed e3m2 (largest 28): as e2m3; row = d*3/4 bytes */
  MJ_KV_E2M1 = 3   /* packed e2m1 (largest 6): code 2j in the low nibble of byte j; row = d/2 bytes */
} mj_kv_format;

/* How the decode call takes Q (T5DecodeRunner's q_mode):
 *   MJ_Q_FP8       — the e4m3 codes and per-(request, KV head) descales
 *                    mj_quantize_q wrote;
 *   MJ_Q_BF16      — the bf16 Q as is (e4m3 KV only, as on the runner page:
 *                    packed e2m3 takes fp8 Q only; the same for e3m2 / e2m1);
 *   MJ_Q_FP8_FUSED — the bf16 Q, quantized by the decode kernel itself with
 *                    mj_quantize_q's recipe (same codes, same descales), so
 *                    the step needs no separate quantize launch. */
typedef enum mj_q_mode { MJ_Q_FP8 = 0, MJ_Q_BF16 = 1, MJ_Q_FP8_FUSED = 2 } mj_q_mode;

/* Element type of the decode output (T5DecodeRunner's out_dtype: bf16 or fp16). */
typedef enum mj_out_dtype { MJ_OUT_BF16 = 0, MJ_OUT_F16 = 1 } mj_out_dtype;

/* Kernel variant of mj_decode_attention. AUTO picks the tensor-core kernel
 * whenever its preconditions hold, else the CUDA-core kernel. */
typedef enum mj_impl { MJ_IMPL_AUTO = 0, MJ_IMPL_SIMT = 1, MJ_IMPL_TCGEN05 = 2 } mj_impl;

#define MJ_KV_TILE 128 /* tokens per KV tile: the unit the plan counts KV in */

/* Human-readable name of a status code (static storage). */
MJ_API const char* mj_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
MJ_API int mj_version(void);

/* ------------------------------------------------------------------------
 * mj_tile_width / mj_slots — the plan's occupancy arithmetic.
 * Source: tile_width() and T5DecodeRunner.n_tiles/.slots on the runner page.
 *   tile_width = next power of two >= n_q, at least 16, at most 32 (fp8 Q);
 *   n_tiles    = ceil(n_q / tile_width);
 *   slots      = max(1, sm_count*ctas_per_sm // (h_k*n_tiles)).
 * ---------------------------------------------------------------------- */
MJ_API int mj_tile_width(int n_q);
MJ_API int mj_slots(int sm_count, int ctas_per_sm, int h_k, int q_len, int h_q);

/* ------------------------------------------------------------------------
 * mj_plan_split_kv — host-only split-KV plan.
 * Source: T5DecodeRunner.plan on the runner page (lens = seq_len + margin;
 * with_reduction = max_splits > 1 && num_seqs < slots, decided by batch SIZE
 * so that a captured graph stays valid), README "A decode step" item 1 (one
 * wave of ctas_per_sm CTAs per SM). The body of plan_split_kv is not on the
 * pages; this implements the reading:
 *   t_b = ceil((seq_lens[b] + margin) / 128)
 *   no reduction:  one row (b, 0, t_b, 0) per request; chunk_tiles = max(1, max t_b)
 *   reduction:     chunk_tiles = smallest c >= 1 with
 *                  sum_b max(1, ceil(t_b/c)) <= slots and max_b ceil(t_b/c) <= max_splits;
 *                  rows (b, s*c, min((s+1)*c, t_b), s) for s < n_splits[b] = max(1, ceil(t_b/c)),
 *                  request-major
 *   padding rows (0, 0, 0, 0) up to pad_to (an empty row: end <= begin).
 *
 * seq_lens_host  [num_seqs] host int32 (exact lengths or an upper bound:
 *                masking always uses the true lengths in device memory).
 * pad_to         number of work rows = the decode grid's x extent; must be
 *                >= max(slots, num_seqs) (T5DecodeRunner.__init__: grid.x is
 *                max(slots, max_num_seqs)), else MJ_ERR_CAPACITY.
 * work_host      [pad_to][4] host int32, written: (request, tile_begin,
 *                tile_end, split).
 * n_splits_host  [num_seqs] host int32, written.
 * chunk_tiles, with_reduction, slots: written scalars (any may be NULL).
 * Deterministic and bit-identical to the CPU oracle's plan.
 * ---------------------------------------------------------------------- */
MJ_API int mj_plan_split_kv(const int32_t* seq_lens_host, int num_seqs, int q_len, int h_q, int h_k,
                     int sm_count, int ctas_per_sm, int max_splits, int margin, int pad_to,
                     int32_t* work_host, int32_t* n_splits_host, int* chunk_tiles,
                     int* with_reduction, int* slots);

/* ------------------------------------------------------------------------
 * mj_plan_upload — copy a host plan into the fixed-address device plan
 * buffers the decode call reads, asynchronously on `stream`.
 * Source: T5DecodeRunner.plan on the runner page (the plan is staged in
 * pinned host memory and copied without blocking into device buffers that
 * keep their addresses, so a captured graph replays new plans).
 * work_host [pad_to][4] and n_splits_host [num_seqs]: the plan
 * mj_plan_split_kv wrote; pinned (page-locked) host memory, which the caller
 * must not overwrite before the copies have run (an event after this call).
 * work_dev / n_splits_dev: device int32 buffers of the same sizes, 16-byte
 * aligned. Enqueues one cudaMemcpyAsync per buffer; MJ_ERR_CUDA if one fails.
 * ---------------------------------------------------------------------- */
MJ_API int mj_plan_upload(const int32_t* work_host, const int32_t* n_splits_host, int32_t* work_dev,
                   int32_t* n_splits_dev, int pad_to, int num_seqs, void* stream);

/* ------------------------------------------------------------------------
 * mj_quantize_q — dynamic per-(request, KV head) e4m3 quantization of Q.
 * Source: T5DecodeRunner.run, fp8-Q branch of the "Q" block (runner page):
 *   x      = float(q) [* q_mul]                      (float32)
 *   amax   = max |x| over (token, GQA head, channel) of (b, g), clamped >= 1e-6f
 *   scale  = amax / 448                              (float32 IEEE division)
 *   code   = e4m3_rne(x / scale)                     (float32 IEEE division)
 *   q_descale[b*h_k + g] = scale
 * Bit-exact with the CPU oracle.
 *
 * q          device bf16, element (b*q_len + t, h, c) at
 *            q[(b*q_len+t)*q_tok_stride + h*q_head_stride + c]; channel stride 1.
 * q_mul      nullable device float32 [h_q][d] (packed KV: K channel scales).
 * q_codes    device uint8 [num_seqs][h_k][q_len*h_r][d], row t*h_r + r
 *            (h_r = h_q/h_k), written.
 * q_descale  device float32 [num_seqs][h_k], written.
 * d is 128 or 256 (T5DecodeRunner asserts head_size % 128 == 0; the library
 * is built for these two), else MJ_ERR_UNSUPPORTED. Padding requests are
 * quantized too (harmless: the decode call never reads them).
 * ---------------------------------------------------------------------- */
MJ_API int mj_quantize_q(const void* q, int64_t q_tok_stride, int64_t q_head_stride, int num_seqs,
                  int q_len, int h_q, int h_k, int d, const float* q_mul, uint8_t* q_codes,
                  float* q_descale, void* stream);

/* ------------------------------------------------------------------------
 * mj_decode_args — everything one decode launch reads and writes.
 * Mirrors the kernel argument list of T5DecodeRunner._launch (runner page):
 * problem shape, block-table row stride, num_pages, num_work, strides, the
 * Q/K/V/block_table/seq_lens/work/n_splits/descale/O/LSE/partial pointers and
 * the softmax scale.
 * ---------------------------------------------------------------------- */
typedef struct mj_decode_args {
  /* problem shape */
  int num_seqs;   /* requests in the batch (real + trailing padding) */
  int q_len;      /* query tokens per request (1 = decode; 1+k = speculative verify) */
  int h_q, h_k;   /* query heads, KV heads; h_q % h_k == 0 */
  int d;          /* head size: 128 or 256 (packed formats at 256: CUDA-core kernel only) */
  int causal;     /* 1: query t sees key j iff j <= seq_len - q_len + t;
                     0: each query token attends to all keys (README "What it does") */
  float softmax_scale;

  /* quantized Q (mj_quantize_q outputs; q_mode MJ_Q_FP8, else unused) */
  const uint8_t* q_codes;  /* [num_seqs][h_k][q_len*h_r][d] */
  const float* q_descale;  /* [num_seqs][h_k] */

  /* paged KV cache: logical (num_pages, page_size, h_k, row) with byte strides */
  int kv_format;           /* mj_kv_format */
  int page_size;           /* tokens per page: 16, 32, 64 or 128 */
  int64_t num_pages;       /* pages in the pool (page ids must be < num_pages) */
  const void* k_cache;
  const void* v_cache;
  int64_t k_stride_page, k_stride_token, k_stride_head;  /* bytes, multiples of 16 */
  int64_t v_stride_page, v_stride_token, v_stride_head;  /* bytes, multiples of 16 */
  /* K/V descales, float32; element (b, g) at ptr[b*seq_stride + g*head_stride]:
     (0,0) per tensor, (0,1) per KV head, (h_k,1) per (request, KV head).
     Packed (e2m3, e3m2, e2m1) KV: the channel scales are folded into q_mul / o_mul and
     these are 1 (_install_fp6_scales, mjolnir/backend.py page). */
  const float* k_descale;
  const float* v_descale;
  int64_t descale_seq_stride, descale_head_stride;

  /* paging */
  const int32_t* block_table;   /* device; page of token j of request b:
                                   block_table[b*block_table_stride + j/page_size] */
  int64_t block_table_stride;
  const int32_t* seq_lens;      /* device [num_seqs]; exact lengths used for masking.
                                   0 = padding request: nothing is written for it. */

  /* plan (mj_plan_split_kv outputs, copied to device) */
  const int32_t* work;          /* device [num_work][4] */
  const int32_t* n_splits;      /* device [num_seqs] */
  int num_work;                 /* = pad_to: the grid's x extent */
  int with_reduction;           /* 1: split partials go to the workspace; call mj_merge_lse */
  int chunk_tiles;              /* tiles per split (plan output) */
  int max_splits;               /* the plan's max_splits (partials indexing) */
  int part_seqs;                /* requests the partial area is sized for (>= num_seqs
                                   when with_reduction; the plan's slots) */

  /* output */
  const float* o_mul;           /* nullable device float32 [h_q][d]: O *= o_mul last */
  void* out;                    /* device bf16 (or fp16, see out_dtype); (b*q_len+t, h, c) at
                                   out[(b*q_len+t)*out_tok_stride + h*out_head_stride + c] */
  int64_t out_tok_stride, out_head_stride;  /* elements, multiples of 8 */
  float* lse;                   /* nullable device float32 [num_seqs][h_k][q_len*h_r]:
                                   natural-log sum of exp(logits) per query row */

  /* caller-owned device workspace (status word + split partials) */
  void* workspace;
  size_t workspace_bytes;

  /* tuning knobs (0 = library default) */
  int impl;          /* mj_impl */
  int kv_stages;     /* KV ring depth of the tensor-core kernel, in K or V tiles (made even,
                        at most 13, and lowered to what shared memory holds); 0 = the
                        deepest even ring up to 6 that keeps two CTAs per SM (4 or 8 query
                        rows per tile at d = 128: 6; 16 rows: 4; d = 256: 2) */
  int evict_first;   /* 1 = L2 evict-first hint on KV loads (KV is read once) */

  int out_dtype;     /* mj_out_dtype of `out` (0 = bf16); rounding to nearest even */

  /* bf16 Q (q_mode MJ_Q_BF16 / MJ_Q_FP8_FUSED): device bf16, (b*q_len+t, h, c)
     at q_bf16[(b*q_len+t)*q_tok_stride + h*q_head_stride + c]; strides in
     elements, multiples of 8. The step is then decode (+ merge) only. */
  int q_mode;        /* mj_q_mode (0 = the fp8 codes above) */
  const void* q_bf16;
  int64_t q_tok_stride, q_head_stride;
  const float* q_mul;  /* MJ_Q_FP8_FUSED: nullable device float32 [h_q][d], as in mj_quantize_q */
} mj_decode_args;

/* ------------------------------------------------------------------------
 * mj_workspace_size — bytes of device workspace a decode step needs.
 * Partials are sized by part_seqs (the plan's slots), not by the batch: the
 * plan only splits when num_seqs < slots (comment above the partial buffers
 * in T5DecodeRunner.__init__). Layout: a 256-byte header holding the device
 * status word, then o_part f32 [part_seqs*max_splits*h_k*n_q_max][d],
 * m_part f32 [..], l_part f32 [..] (n_q_max = max_q_len*h_q/h_k).
 * ---------------------------------------------------------------------- */
MJ_API int mj_workspace_size(int part_seqs, int max_splits, int max_q_len, int h_q, int h_k, int d,
                      size_t* bytes);

/* Zero the workspace status word (enqueued on `stream`). Call once after
 * allocating the workspace. */
MJ_API int mj_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Read and clear the workspace status word. SYNCHRONISES `stream` (a test and
 * debugging aid, not for the hot path). *device_status = 0 means no kernel
 * recorded an anomaly; otherwise a bit mask (1: page id out of range,
 * 2: a bounded wait timed out, 4: a work row outside the partial area). Returns MJ_ERR_DEVICE_CHECK when non-zero. */
MJ_API int mj_workspace_status(void* workspace, void* stream, uint32_t* device_status);

/* ------------------------------------------------------------------------
 * mj_decode_attention — paged decode attention over the plan's work rows.
 * Source: README "A decode step" item 3 (stream KV pages into a shared-memory
 * ring, tensor-core S and O, online softmax), T5DecodeRunner._launch/run.
 * Reads each valid KV row once. For a work row (b, tb, te, s) and KV head g
 * it covers keys [tb*128, min(te*128, seq_lens[b])) and all q_len*h_r query
 * rows of (b, g):
 *   - if !with_reduction or n_splits[b] == 1: writes the final output (bf16 or fp16, out_dtype)
 *     O * v_descale * o_mul and, if lse != NULL, the row LSE;
 *   - else writes its normalised partial (O~, m, l) into the workspace.
 * Rows of requests with seq_lens[b] == 0 and empty work rows write nothing.
 * Grid: num_work x h_k x n_row_tiles CTAs (the tensor-core kernel orders
 * them KV head fastest), fixed by the arguments.
 * Accuracy: the tensor-core kernel scales the softmax weights p to the row's
 * running max (p <= 2^8.6) and carries each in e4m3 terms: hi = e4m3(p) and
 * lo = e4m3(p - hi), within max(2^-8 p, 2^-10) of p; where weights below 1/4
 * are many (more than 1024 per row in a CTA's key range) it adds, for them,
 * the same split of (p - hi - lo) * 2^10 weighed 2^-10, which brings every
 * weight within max(2^-8 p, 2^-20). The row sum l adds the p themselves. So
 * keys down to 27 binades (about 19 nats) below the row's max keep their
 * weight, and the output of a row of N keys is off by at most
 * (2^-7 + N * 2^-28) * max|V|. MJ_IMPL_SIMT keeps the weights in float32.
 * Ordering: with q_mode MJ_Q_FP8 the tensor-core launch may begin before the
 * preceding kernel on `stream` has finished (programmatic dependent launch:
 * only its Q reads wait for that kernel), so that kernel must be the
 * mj_quantize_q call that wrote q_codes, with nothing enqueued in between;
 * the other Q modes are stream-ordered for everything the kernel reads: its
 * CTAs may start early, but before the preceding kernel has finished they
 * only ask L2 to prefetch their first KV tiles (aimed with the plan and
 * block table as they stand; a prefetch returns no data), and without a split
 * they let the next kernel on `stream` launch early in the same way.
 * ---------------------------------------------------------------------- */
MJ_API int mj_decode_attention(const mj_decode_args* args, void* stream);

/* Which kernel mj_decode_attention runs for these arguments: *impl is set to
 * MJ_IMPL_TCGEN05 or MJ_IMPL_SIMT. Validates like that call and launches
 * nothing; MJ_ERR_UNSUPPORTED when args->impl asks for the tensor-core kernel
 * and it cannot take the arguments. */
MJ_API int mj_decode_kernel(const mj_decode_args* args, int* impl);

/* ------------------------------------------------------------------------
 * mj_merge_lse — combine split-KV partials by log-sum-exp.
 * Source: README "A decode step" item 4 (a separate, small kernel merges
 * the split-KV partials by their LSE). For each request b with n_splits[b] > 1 and
 * seq_lens[b] > 0, KV head g and query row:
 *   M = max_s m_s;  w_s = 2^(m_s - M) * l_s (0 for empty splits);
 *   O = sum_s w_s O~_s / sum_s w_s, times v_descale and o_mul, rounded to the output type
 *   (bf16 or fp16, out_dtype; to nearest even).
 * Splits whose first key is at or past seq_lens[b] are empty and skipped.
 * A no-op when args->with_reduction == 0. Same argument struct as
 * mj_decode_attention (it reads the partials that call left in the workspace).
 * ---------------------------------------------------------------------- */
MJ_API int mj_merge_lse(const mj_decode_args* args, void* stream);

/* ------------------------------------------------------------------------
 * mj_decode_attention_noalloc — mj_decode_attention followed by mj_merge_lse,
 * with the split-KV partials in scratch memory compiled into the library
 * instead of a caller workspace. The pages have no counterpart for this call.
 *
 * For callers that cannot allocate device memory: an engine that reserves
 * almost all of HBM for its KV-cache pool at start-up and allows no later
 * cudaMalloc, or a plugin inside a framework whose caching allocator owns
 * device memory (a raw cudaMalloc/cudaFree would bypass it and synchronise
 * the device). Such a caller still passes every input and output; only
 * args->workspace and args->workspace_bytes are ignored.
 *
 * The scratch is a fixed MJ_NOALLOC_SCRATCH_BYTES array (16 MiB) that every
 * GPU loading the library holds until the process exits. A plan whose
 * partials need more (mj_workspace_size(part_seqs, max_splits, ...) above the
 * limit) is rejected with MJ_ERR_CAPACITY before anything is enqueued. The
 * first call on a device looks up the array's device address and zeroes its
 * status header on the caller's stream; make that first call before any
 * stream capture. All calls share the array and it keeps the last call's contents:
 * calls whose kernels overlap on the GPU race on it, so issue them in order
 * on one stream. The kernels record anomalies (a page id out of range, a
 * bounded wait that timed out, a work row outside the partial area) in a
 * status word in the scratch header; mj_noalloc_status reads it.
 * ---------------------------------------------------------------------- */
#define MJ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
MJ_API int mj_decode_attention_noalloc(const mj_decode_args* args, void* stream);

/* Read and clear the status word of the current device's allocation-free
 * scratch, like mj_workspace_status does for a caller workspace: SYNCHRONISES
 * `stream` (a test and debugging aid, not for the hot path); *device_status = 0
 * means no anomaly, else the same bit mask; returns MJ_ERR_DEVICE_CHECK when
 * it is non-zero. Called before any mj_decode_attention_noalloc on the device,
 * it performs that call's first-call set-up and reads 0. */
MJ_API int mj_noalloc_status(void* stream, uint32_t* device_status);

/* ------------------------------------------------------------------------
 * mj_write_kv — the KV-cache write that precedes a decode step: quantize the
 * new tokens' K and V rows and scatter them into the paged caches at
 * slot_mapping. Source: MjolnirImpl.do_kv_cache_update / _write_kv on the
 * mjolnir/backend.py page (the e4m3 write takes the layer's k/v scale; the
 * packed e2m3 write takes the per-(KV head, channel) scales that
 * _install_fp6_scales applies when the cache is written).
 *
 * For token t and KV head g with s = slot_mapping[t] >= 0, the row goes to
 * page s / page_size, row s % page_size of the cache (the decode call's
 * layout and strides):
 *   e4m3: code[c] = e4m3(x[c] / scale)      scale = k_scale[0] (per tensor)
 *                                           or k_scale[g] (scale_per_head)
 *   e2m3: code[c] = e2m3(x[c] / k_scale[g*d + c]), packed 4 codes per 3 bytes
 *   e3m2, e2m1: likewise with their own code and packing (mj_kv_format)
 * x is the bf16 input widened to float32; the division is IEEE float32 and
 * the rounding to the cache format is to nearest, ties to even, saturating
 * (448 / 7.5 / 28 / 6). Likewise for V with v_scale. A negative slot marks a padding
 * token: nothing is written for it. A slot at or past num_pages*page_size is
 * skipped and, if status != NULL, bit 1 of *status is set.
 *
 * Alignment: key/value 16-byte aligned with token/head strides that are
 * multiples of 8 elements; cache bases 16-byte aligned with byte strides that
 * are multiples of 16. The caches are written in place; every byte outside
 * the written rows keeps its value. The call enqueues one kernel on `stream`.
 * ---------------------------------------------------------------------- */
typedef struct mj_write_kv_args {
  int num_tokens;             /* rows in key / value (0: nothing to do) */
  int h_k, d;                 /* KV heads; head size (128 or 256) */
  const void* key;            /* device bf16; (t, g, c) at key[t*key_tok_stride + g*key_head_stride + c] */
  const void* value;          /* device bf16; likewise with the value strides */
  int64_t key_tok_stride, key_head_stride;      /* elements */
  int64_t value_tok_stride, value_head_stride;  /* elements */
  const int64_t* slot_mapping;  /* device [num_tokens] */

  int kv_format;              /* mj_kv_format */
  int page_size;              /* tokens per page: 16, 32, 64 or 128 */
  int64_t num_pages;
  void* k_cache;
  void* v_cache;
  int64_t k_stride_page, k_stride_token, k_stride_head;  /* bytes */
  int64_t v_stride_page, v_stride_token, v_stride_head;  /* bytes */

  const float* k_scale;       /* device float32: e4m3 [1] or [h_k]; packed formats [h_k][d] */
  const float* v_scale;
  int scale_per_head;         /* e4m3 only: 1 = one scale per KV head, 0 = per tensor */

  uint32_t* status;           /* nullable device word (see above) */
} mj_write_kv_args;

MJ_API int mj_write_kv(const mj_write_kv_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MJ_H */
