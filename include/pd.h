/*
 * pd.h - C ABI of libpd.so: paged split-KV decode attention on GB300 (sm_103a).
 *
 * Every operation here is one step of single-token (decode) attention for a
 * batch of sequences whose keys and values live in a paged KV cache read
 * through a block table, with grouped-query heads, cut into split-KV
 * partials that a log-sum-exp combine merges. The passages each call follows
 * are cited beside it:
 *   [metrale]   docs.metrale.ai, "prefill_attn_b.rs" (launchers for the NVFP4
 *               cache write, `bf16_absmax`, `paged_decode_attn_splitk_*` and
 *               `paged_decode_attn_reduce_*`);
 *   [AstrAI]    "ViperEkura/AstrAI csrc/tests" commit log (split-KV decode
 *               with o_part / ml_part and a single combine kernel,
 *               compute_num_splits, int32 indices, divisibility checks);
 *   [pegainfer] pegainfer issue 1008 (paged decode / split-KV decode units).
 *
 * Conventions for every call:
 *   - Pointers named as device memory must be device pointers (or managed
 *     memory) owned by the caller; the library keeps no reference after the
 *     call returns, allocates nothing and never synchronises.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued on it, in order.
 *   - Every device pointer must be 16-byte aligned.
 *   - Return value: PD_OK, or a pd_status code; nothing throws. Argument
 *     errors are reported before anything is enqueued. PD_ERR_CUDA means a
 *     launch failed (cudaGetLastError was not cudaSuccess).
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16).
 *
 * Cache layouts (per K cache and per V cache; kv_dtype selects the form):
 *   PD_KV_BF16      page = bf16 [block_size][num_kv_heads][head_dim]
 *                   ([metrale] "the cache is [blocks, block_size, kv_heads,
 *                   head_dim] and the kernel computes the page stride").
 *   PD_KV_FP8_E4M3  page = E4M3 bytes [block_size][num_kv_heads][head_dim];
 *                   value = decode(byte) * k_scale (or v_scale), per-tensor
 *                   fp32 scales ([metrale] `paged_decode_attn_splitk_fp8`,
 *                   k_scale / v_scale / cache_stride).
 *   PD_KV_NVFP4     page = data section E2M1 nibbles
 *                   [num_kv_heads][block_size][head_dim/2] (element 2i in the
 *                   low nibble) followed by the scale section, one E4M3 byte
 *                   per 16 elements [num_kv_heads][block_size][head_dim/16];
 *                   the page stride is rounded up to a multiple of 128 bytes
 *                   ([metrale] `reshape_and_cache_nvfp4`: "E2M1 values with
 *                   one E4M3 scale per 16", block_stride_bytes,
 *                   data_section_bytes). The order inside each section is
 *                   this library's choice; the pages leave it open.
 *   Slot s of the pool is page s / block_size, row s % block_size.
 */
#ifndef PD_H_
#define PD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum pd_status {
  PD_OK = 0,
  PD_ERR_INVALID_ARG = 1,         /* null / misaligned pointer, bad size or shape */
  PD_ERR_UNSUPPORTED = 2,         /* head_dim, block_size, group size or dtype not built */
  PD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < pd_decode_workspace_bytes(...) */
  PD_ERR_CUDA = 4                 /* a CUDA runtime call or kernel launch failed */
};

/* KV cache forms. */
enum pd_kv_dtype { PD_KV_BF16 = 0, PD_KV_FP8_E4M3 = 1, PD_KV_NVFP4 = 2 };

/* Device-side status bits, accumulated by the kernels (see pd_device_status). */
enum pd_device_flag {
  PD_DEV_BAD_PAGE = 1,    /* a block_tables entry was < 0 or >= num_blocks: page skipped */
  PD_DEV_BAD_SEQ_LEN = 2, /* seq_lens[b] < 0 or > max_blocks_per_seq*block_size: clamped */
  PD_DEV_BAD_SLOT = 4,    /* slot_mapping[t] >= num_blocks*block_size: token skipped */
  PD_DEV_TIMEOUT = 8,     /* a bounded wait inside a kernel gave up: that output is invalid */
  PD_DEV_BAD_PLAN = 16,   /* a balanced-plan entry was out of range: that piece skipped */
  PD_DEV_BAD_SMEM = 32    /* a kernel found its shared memory off the 1024-byte boundary
                             its swizzled tiles need: it wrote nothing */
};

/* Human-readable name of a pd_status value (static string, never NULL). */
const char* pd_status_string(int status);

/* Bytes of one K (or one V) cache of num_blocks pages in the given form.
 * Returns 0 for an unsupported combination. Host-only, no CUDA call. */
size_t pd_cache_bytes(int32_t kv_dtype, int64_t num_blocks, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_dim);

/* Bytes of one page (the page stride) in the given form; 0 if unsupported. */
size_t pd_page_bytes(int32_t kv_dtype, int32_t block_size, int32_t num_kv_heads,
                     int32_t head_dim);

/* Write (and quantise) each token's K and V rows into the paged caches at
 * slot_mapping[t] ([metrale] `reshape_and_cache_nvfp4`: "Write each token's
 * K and V into the paged NVFP4 cache at its slot_mapping slot", extended to
 * the BF16 and FP8 forms that the decode launchers read).
 *   key, value    device bf16 [num_tokens][num_kv_heads][head_dim], contiguous.
 *   k_cache,      device caches of pd_cache_bytes(kv_dtype, num_blocks, ...)
 *   v_cache       bytes each; only the slots named by slot_mapping change.
 *   slot_mapping  device int32 [num_tokens]; a negative slot skips the token
 *                 (padding); a slot >= num_blocks*block_size is skipped and
 *                 flagged PD_DEV_BAD_SLOT.
 *   BF16 copies the bit patterns. FP8 stores E4M3(float(x) / scale) with
 *   IEEE fp32 division, round to nearest even and saturation to +-448
 *   (NaN -> 0x7F|sign). NVFP4 stores, per 16 consecutive elements of a
 *   (token, head) row, scale = E4M3(amax / 6) with amax = max |x| (NaN
 *   skipped) and codes E2M1(float(x) / decode(scale)) rounded to nearest
 *   even and saturated to +-6 (NaN -> +-6); a group whose scale decodes to 0
 *   stores +0 codes. k_scale / v_scale are read only for FP8 and must then be
 *   finite and > 0.
 * head_dim in {64, 128, 256, 512}; block_size in {16, 32}; num_tokens >= 0. */
int pd_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int32_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         int32_t kv_dtype, float k_scale, float v_scale, void* stream);

/* Max |x| over n bf16 values, folded into *out_max with an atomic max
 * ([metrale] `bf16_absmax`: "The caller zeroes out_max first"). NaN values
 * are skipped. data: device bf16 [n]; out_max: device float, caller-zeroed.
 * The first half of FP8 calibration; pd_fp8_scale / pd_fp8_scales_from_absmax
 * turn the maximum into the per-tensor scale. */
int pd_absmax_bf16(const void* data, int64_t n, float* out_max, void* stream);

/* FP8 calibration scale of one tensor from its absmax ([metrale] `bf16_absmax`:
 * the FP8 KV calibration runs it before each K / V pair; the scale maps the
 * tensor's largest magnitude onto E4M3's largest finite value, 448):
 * absmax / 448 in IEEE fp32 division, or 1.0 when absmax is not > 0 (an
 * all-zero tensor; NaN). Host only, no CUDA call. Pass the result as
 * pd_reshape_and_cache's k_scale / v_scale and pd_decode's. */
float pd_fp8_scale(float absmax);

/* The same on the device: scales[i] = pd_fp8_scale(absmax[i]) for i < count,
 * with absmax the outputs of pd_absmax_bf16 (device float [count]) and scales
 * device float [count] (4-byte aligned). Enqueued on `stream`, no
 * synchronisation: a caller reads the scales back once, after calibration. */
int pd_fp8_scales_from_absmax(const float* absmax, float* scales, int32_t count, void* stream);

/* Workspace bytes that pd_decode / pd_decode_partial need for num_splits
 * partials: per (sequence, q head, split) head_dim fp32 values of the
 * normalised partial output plus its running max m and sum l ([metrale]:
 * "The workspace is F32 [head_dim values, m, l] per split"). */
size_t pd_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t num_splits);

/* Split count chosen from the SM count of `device` and the number of page
 * tiles ([AstrAI] compute_num_splits "only use base_blocks and
 * tiles_total"; short sequences get more splits). Returns S >= 1, or a
 * negative pd_status on error. Depends only on the shapes, never on the
 * contents of seq_lens, so it needs no device read. */
int pd_choose_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                         int32_t block_size, int32_t sliding_window, int32_t head_dim,
                         int32_t kv_dtype, int device);

/* The same choice with the SM count given (no CUDA call): one CTA per
 * (sequence, kv head, split), S chosen so that the grid is about one wave of
 * resident CTAs when every sequence is at its maximum length. */
int pd_plan_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                       int32_t block_size, int32_t sliding_window, int32_t head_dim,
                       int32_t kv_dtype, int32_t num_sms);

/* Split count for known sequence lengths (host array seq_lens[num_seqs], as a
 * serving scheduler holds them): replays the launch in block order onto the
 * resident CTA slots with a per-CTA start-up cost, adds the partial and
 * combine traffic, and returns the S with the smallest estimated time.
 * Host-only, no CUDA call; returns S >= 1 or a negative pd_status. */
int pd_plan_num_splits_for_lengths(const int32_t* seq_lens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t max_blocks_per_seq, int32_t block_size,
                                   int32_t sliding_window, int32_t head_dim, int32_t kv_dtype,
                                   int32_t num_sms);

/* One decode step: split-KV partials then the log-sum-exp combine.
 * out[b, h, :] = bf16( sum_j e_j v_j / sum_j e_j ), e_j = exp(s_j - max s),
 * s_j = scale * (q[b, h, :] . k_j), over the keys j of sequence b inside the
 * window, k_j / v_j read from page block_tables[b, j / block_size], row
 * j % block_size, kv head h / (num_q_heads / num_kv_heads).
 *   q             device bf16 [num_seqs][num_q_heads][head_dim], contiguous.
 *   k_cache,      device caches in the kv_dtype form (layout above).
 *   v_cache
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; only the
 *                 entries of pages holding keys in the window are read.
 *   seq_lens      device int32 [num_seqs], 0 <= L <= max_blocks_per_seq *
 *                 block_size (L = 0 writes a zero row).
 *   out           device bf16 [num_seqs][num_q_heads][head_dim].
 *   scale         score multiplier, usually 1/sqrt(head_dim).
 *   num_splits    0 = pd_choose_num_splits on the current device, else S.
 *   sliding_window  0 = off; W > 0 keeps keys j with (L-1) - j < W.
 *   k_scale, v_scale  FP8 per-tensor scales (ignored for other forms).
 *   workspace     device scratch of >= pd_decode_workspace_bytes(num_seqs,
 *                 num_q_heads, head_dim, S) bytes; its contents on entry do
 *                 not matter.
 * ([metrale] `paged_decode_attn_splitk_{nvfp4,fp8,bf16}` +
 * `paged_decode_attn_reduce_{nvfp4,fp8}`; [AstrAI] split-KV paged decode
 * with o_part / ml_part and one combine kernel.)
 * Supported: head_dim in {64, 128, 256, 512} (NVFP4: all of them);
 * block_size in {16, 32}; num_q_heads % num_kv_heads == 0 with a group of
 * at most 16; 1 <= S <= 1024. */
int pd_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* seq_lens, void* out, int32_t num_seqs, int32_t num_q_heads,
              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
              int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t num_splits,
              int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
              void* workspace, size_t workspace_bytes, void* stream);

/* pd_decode with q read from and out written to rows that need not be
 * packed, as in a fused QKV buffer ([metrale] `q_stride`; [AstrAI]
 * "stride-based addressing for Q/KV/O"): sequence b's q heads are the
 * num_q_heads * head_dim contiguous bf16 values at q + b * q_stride, and its
 * output heads go to out + b * out_stride. Both strides are in elements,
 * >= num_q_heads * head_dim and a multiple of 8 (16-byte aligned rows);
 * PD_ERR_INVALID_ARG otherwise. Everything else is as pd_decode. */
int pd_decode_strided(const void* q, int64_t q_stride, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, void* out,
                      int64_t out_stride, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                      int32_t num_splits, int32_t sliding_window, int32_t kv_dtype,
                      float k_scale, float v_scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/* pd_decode writing the output as E4M3 bytes instead of bf16 (the "E4M3
 * output variant" that [AstrAI] lists beside stride-based addressing; the
 * pages define no output scale or rounding, so this library's reading is):
 *   out[b, h, d] = E4M3(o[b, h, d] / out_scale)
 * with o the fp32 attention output (before any bf16 rounding), out_scale a
 * per-tensor fp32 scale (finite, > 0; PD_ERR_INVALID_ARG otherwise), IEEE
 * fp32 division and pd_reshape_and_cache's E4M3 rules (nearest, ties to
 * even, saturation to +-448, the sign of a zero kept). A code c stands for
 * decode(c) * out_scale. out: device uint8 [num_seqs][num_q_heads][head_dim],
 * 16-byte aligned. Every sequence's partials go through the workspace (no
 * direct single-split write), so workspace_bytes >=
 * pd_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, S). Everything
 * else as pd_decode. */
int pd_decode_e4m3_out(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens, void* out,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                       int64_t num_blocks, float scale, int32_t num_splits,
                       int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                       float out_scale, void* workspace, size_t workspace_bytes, void* stream);

/* The first half of pd_decode alone: writes the S partials (O_s normalised,
 * m_s, l_s) of every (sequence, q head) to the workspace ([metrale]: "each
 * block writes its partial output and softmax state to workspace"). Same
 * arguments as pd_decode, with num_splits >= 1 required. Splits that hold
 * no key of a sequence are not written. */
int pd_decode_partial(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks,
                      float scale, int32_t num_splits, int32_t sliding_window, int32_t kv_dtype,
                      float k_scale, float v_scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/* The second half of pd_decode alone: merges the partials that
 * pd_decode_partial wrote into out, M = max_s m_s, w_s = l_s exp(m_s - M),
 * out = bf16(sum_s w_s O_s / max(sum_s w_s, 1e-20)) ([metrale] `paged_decode
 * _attn_reduce_fp8`: "Combine split-K partials into the BF16 output"; it
 * reads seq_lens to know how many splits of each sequence hold keys).
 * Arguments must match the pd_decode_partial call that filled workspace. */
int pd_decode_combine(const void* workspace, size_t workspace_bytes, const int32_t* seq_lens,
                      void* out, int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_blocks_per_seq, int32_t num_splits,
                      int32_t sliding_window, void* stream);

/* ---- Balanced decode: a host-made plan that gives every CTA equal work ----
 *
 * pd_decode splits every sequence into the same S splits, so CTAs get unequal
 * work when lengths differ and the grid runs in several generations. A
 * serving scheduler already holds the lengths on the host; from them
 * pd_balanced_plan cuts the line of all (sequence, kv head) key ranges, laid
 * end to end in sequence-major order, into one equal share of pages per
 * resident CTA (the split-KV partition of [metrale] `paged_decode_attn_splitk_*`
 * with per-head, length-dependent split points). A share that crosses a head's
 * range boundary holds several "pieces"; each piece gets its own partial
 * (O, m, l), merged by the same log-sum-exp combine ([metrale]
 * `paged_decode_attn_reduce_*`). Results equal pd_decode's up to fp32
 * summation order. */

/* Which schedule to run for these host lengths: 1 if the balanced one is
 * expected to be faster than pd_decode with pd_plan_num_splits_for_lengths'
 * split count, 0 if not, a negative pd_status on bad arguments. Host only.
 * It compares the split planner's estimated makespan with an equal share per
 * CTA plus a measured per-tile premium of the balanced kernel (about 5 %) and
 * its per-piece cost: lengths that differ favour the balanced schedule,
 * equal lengths the split one. */
int pd_prefer_balanced(const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t max_blocks_per_seq, int32_t block_size,
                       int32_t sliding_window, int32_t head_dim, int32_t kv_dtype,
                       int32_t num_sms);

/* Upper bound of the plan bytes for num_seqs sequences, num_kv_heads heads and
 * a device with num_sms SMs (host only). */
size_t pd_balanced_plan_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t num_sms);

/* Build the plan on the host from host seq_lens[num_seqs] (clamped to
 * [0, max_blocks_per_seq * block_size], windowed like pd_decode).
 *   plan          host buffer, 16-byte aligned, of plan_bytes >=
 *                 pd_balanced_plan_bytes; copy it to the device before
 *                 pd_decode_balanced (its bytes, as written, are the device
 *                 plan). The plan is valid only for these lengths: build a new
 *                 one whenever a length changes.
 *   num_ctas, num_pieces  out: pass them to pd_decode_balanced.
 *   workspace_bytes       out: the workspace pd_decode_balanced needs.
 * Returns PD_OK, PD_ERR_INVALID_ARG / PD_ERR_UNSUPPORTED on bad shapes, or
 * PD_ERR_WORKSPACE_TOO_SMALL if plan_bytes is short. No CUDA call. */
int pd_balanced_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t max_blocks_per_seq, int32_t sliding_window, int32_t kv_dtype,
                     int32_t num_sms, void* plan, size_t plan_bytes, int32_t* num_ctas,
                     int32_t* num_pieces, size_t* workspace_bytes);

/* One decode step over a balanced plan: the partial kernel (one CTA per plan
 * share, pieces in order; a head covered by one piece is written to out
 * directly) and then the combine, which also writes the zero rows of empty
 * sequences. Arguments as pd_decode, with
 *   plan, plan_bytes       the device copy of pd_balanced_plan's output.
 *   num_ctas, num_pieces   pd_balanced_plan's outputs for that plan.
 *   workspace              device scratch of >= the planner's workspace_bytes;
 *                          contents on entry do not matter.
 * seq_lens is not an argument: the plan carries each piece's key range.
 * Plan entries out of range are skipped and raise PD_DEV_BAD_PLAN in the
 * device status word. No allocation, no synchronisation. */
int pd_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const void* plan, size_t plan_bytes,
                       void* out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                       int64_t num_blocks, float scale, int32_t sliding_window,
                       int32_t kv_dtype, float k_scale, float v_scale, int32_t num_ctas,
                       int32_t num_pieces, void* workspace, size_t workspace_bytes,
                       void* stream);

/* pd_decode_balanced with strided q and output rows (as for pd_decode_strided). */
int pd_decode_balanced_strided(const void* q, int64_t q_stride, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const void* plan, size_t plan_bytes, void* out,
                               int64_t out_stride, int32_t num_seqs,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, int32_t sliding_window,
                               int32_t kv_dtype, float k_scale, float v_scale, int32_t num_ctas,
                               int32_t num_pieces, void* workspace, size_t workspace_bytes,
                               void* stream);

/* The two halves of pd_decode_balanced, with its arguments: the partial
 * kernel alone (writes the workspace partials and the rows of heads one
 * piece covers), then the combine alone (reads the same workspace and plan).
 * For timing each kernel on its own; pd_decode_balanced launches both. */
int pd_decode_balanced_partial(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const void* plan, size_t plan_bytes,
                               void* out, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                               int32_t sliding_window, int32_t kv_dtype, float k_scale,
                               float v_scale, int32_t num_ctas, int32_t num_pieces,
                               void* workspace, size_t workspace_bytes, void* stream);
int pd_decode_balanced_combine(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const void* plan, size_t plan_bytes,
                               void* out, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                               int32_t sliding_window, int32_t kv_dtype, float k_scale,
                               float v_scale, int32_t num_ctas, int32_t num_pieces,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Size of the workspace array that pd_decode_static_ws uses (8 MiB). */
#define PD_STATIC_WORKSPACE_BYTES (8u << 20)

/* pd_decode for callers that cannot allocate device memory. None of the
 * three pages has a counterpart of this call: it exists for code that only
 * receives its input and output buffers - an operator running inside another
 * runtime that owns all device memory, or a caller with a fixed memory budget
 * - and so has no way to provide pd_decode's workspace.
 * Arguments and results are those of pd_decode without `workspace` and
 * `workspace_bytes`: the split partials go to a fixed array of
 * PD_STATIC_WORKSPACE_BYTES that libpd.so reserves on every device that loads
 * it, for the life of the process.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 *     call. The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     outside any stream capture.
 *   - Returns PD_ERR_WORKSPACE_TOO_SMALL when pd_decode_workspace_bytes for
 *     the split count (num_splits, or the automatic choice when 0) exceeds
 *     PD_STATIC_WORKSPACE_BYTES.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents (nothing in it needs to start at zero). Calls whose
 *     work overlaps on the GPU - on different streams, or from different
 *     host threads - race on it: serialise them. */
int pd_decode_static_ws(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* seq_lens, void* out,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                        int64_t num_blocks, float scale, int32_t num_splits,
                        int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                        void* stream);

/* Paged prefill (chunked prefill) attention over the same paged cache:
 * several query tokens per sequence. pegainfer issue 1008 names the unit
 * (`prefill_paged_launch` over the paged-KV view); the AstrAI "csrc/tests"
 * log gives its interface: one causal offset (-1 = off, >= 0 = the first
 * query position), stride addressing for Q and O, the paged KV source.
 *   q, out      bf16; query row i (i in [0, cu_q[num_seqs])) holds the
 *               num_q_heads x head_dim values of one token at element
 *               i * q_stride / i * out_stride (0 = packed, num_q_heads *
 *               head_dim; otherwise at least that and a multiple of 8).
 *   cu_q        int32 [num_seqs + 1], device: sequence b owns query rows
 *               [cu_q[b], cu_q[b+1]), its q_len_b newest tokens.
 *   seq_lens    int32 [num_seqs], device: L_b keys in the cache, the new
 *               tokens already written (pd_reshape_and_cache), q_len_b <= L_b.
 *   max_q_len   host int: the largest q_len_b; the grid covers that many
 *               tokens per sequence (a longer one raises PD_DEV_BAD_SEQ_LEN).
 *   causal      != 0: query i of sequence b sits at position L_b - q_len_b + i
 *               (the causal offset of the sequence is L_b - q_len_b) and sees
 *               keys j <= its position; 0: every query sees all L_b keys.
 *   sliding_window  W > 0 keeps keys j with position - j < W; 0 = off.
 * Scores, softmax and the bf16 output follow pd_decode (scale after the dot
 * product, 1e-20 guard). Cache (all three forms, with k_scale / v_scale for
 * FP8), block tables, scale, status codes and device flags as in pd_decode
 * ([AstrAI]: prefill kernels templated on the paged KV source). Supported:
 * head_dim 64, 128 or 256, block_size 16 or 32, G = num_q_heads /
 * num_kv_heads <= 16; anything else returns PD_ERR_UNSUPPORTED. No
 * workspace: each query tile writes its rows. BF16 caches run on the tcgen05
 * tensor cores (accumulators in TMEM; at head_dim 64 and 128 two 128-row
 * query tiles share each CTA's K/V stages); FP8 and NVFP4 caches on mma.sync
 * tiles, each stage widened once to f16 (exact) before its MMAs.
 * Device pointers owned by the caller, 16-byte aligned; enqueued on `stream`,
 * never synchronises. */
int pd_prefill(const void* q, int64_t q_stride, const int32_t* cu_q, const void* k_cache,
               const void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
               void* out, int64_t out_stride, int32_t num_seqs, int32_t max_q_len,
               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
               int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t causal,
               int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
               void* stream);

/* ---- Cross-check kernels ----
 * Independent second implementations of two steps, kept to test the fast
 * kernels against: same arguments, same results up to fp32 summation order.
 * They are slower and never chosen by the calls above. */

/* pd_decode with the split-KV partials computed on CUDA cores (one warp per
 * key for the scores, plain fp32 loops for P V) instead of the tensor-core
 * kernel; every partial goes through the workspace and the combine. */
int pd_decode_crosscheck(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, void* out,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                         int64_t num_blocks, float scale, int32_t num_splits,
                         int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                         void* workspace, size_t workspace_bytes, void* stream);

/* pd_prefill on mma.sync tensor-core tiles (64 query rows per CTA) instead of
 * the tcgen05 kernel. Same arguments and support as pd_prefill (for FP8 and
 * NVFP4 caches pd_prefill runs this kernel itself). */
int pd_prefill_crosscheck(const void* q, int64_t q_stride, const int32_t* cu_q,
                          const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          const int32_t* seq_lens, void* out, int64_t out_stride,
                          int32_t num_seqs, int32_t max_q_len, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                          int32_t causal, int32_t sliding_window, int32_t kv_dtype,
                          float k_scale, float v_scale, void* stream);

/* ---- Test hooks ----
 * For the library's own tests; a serving process has no reason to call them. */

/* Run the cache write's own device encoders on fp32 bit patterns:
 * codes[i] = code of the float whose bits are first_bits + i (mod 2^32), for
 * i < count <= 2^32; format 0 = E4M3 (the FP8 cache, rules of
 * pd_reshape_and_cache), 1 = E2M1 (the NVFP4 values). codes: device uint8
 * [count]. Lets a test compare the encoders with a reference over every fp32
 * input, including quotients no bf16 input and scale produce. */
int pd_test_encode(int32_t format, uint32_t first_bits, int64_t count, uint8_t* codes,
                   void* stream);

/* Set the limit (ns) of the decode partial kernels' consumer-side waits for a
 * stage of keys, for calls made after it; 0xFFFFFFFF restores the default
 * (2 s). Returns the previous limit. A test sets it to 0 so that those waits
 * run out at once, to see the bounded-wait path report PD_DEV_TIMEOUT and the
 * kernel end normally: a consumer warp that gives up stops handing stages
 * back and raises its CTA's abort word; the producer then issues nothing more
 * and waits for every copy it already issued before the CTA ends. The outputs
 * of such a call are invalid. Process-wide, not thread-safe against
 * concurrent decode calls. */
uint32_t pd_test_set_consumer_wait_ns(uint32_t ns);

/* Read (and, if reset != 0, clear) the pd_device_flag bits that kernels on
 * the current device have raised since the last reset. Synchronises the
 * device (cudaMemcpyFromSymbol): a debugging call, not for the hot path. */
int pd_device_status(int32_t* flags, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* PD_H_ */
