// Device helpers shared by the libpd.so kernels: bf16 / E4M3 / E2M1 codecs,
// split geometry and the argument blocks passed to the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pd.h"

namespace pd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxGroup = 16;

// ---------------------------------------------------------------------------
// bf16
__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// the two bf16 halves of a 32-bit word, low half first
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// E4M3 (OCP "E4M3FN": bias 7, no Inf, S.1111.111 = NaN, max 448).
// Encoder: round to nearest even on the E4M3 grid, finite overflow and Inf
// saturate to +-448, NaN -> 0x7F | sign, the sign of a zero result is kept.
// Written on the fp32 bit fields; needs IEEE denormal support (no -ftz).
__device__ __forceinline__ uint32_t e4m3_encode(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t sign = (u >> 24) & 0x80u;
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return 0x7Fu | sign;    // NaN
  if (a >= 0x43E00000u) return 0x7Eu | sign;   // |x| >= 448 (and Inf): saturate
  if (a < 0x3C800000u) {                       // |x| < 2^-6: multiples of 2^-9
    // exact scaling by 2^9, then round to the nearest integer, ties to even;
    // 8 is the smallest normal 2^-6, whose code is also 8
    const uint32_t n = __float2uint_rn(__uint_as_float(a) * 512.0f);
    return n | sign;
  }
  int e = static_cast<int>(a >> 23) - 127;     // -6 .. 8
  uint32_t keep = (a >> 20) & 0x7u;            // top 3 mantissa bits
  const uint32_t rest = a & 0xFFFFFu;          // the 20 bits rounded away
  if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) ++keep;
  if (keep == 8u) {
    keep = 0u;
    ++e;
  }
  return (static_cast<uint32_t>(e + 7) << 3) | keep | sign;
}

__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  const uint32_t sign = (c & 0x80u) << 24;
  const uint32_t ex = (c >> 3) & 0xFu;
  const uint32_t man = c & 0x7u;
  if (ex == 0xFu && man == 0x7u) return __uint_as_float(0x7FC00000u | sign);
  if (ex == 0u) return __uint_as_float(sign | __float_as_uint(static_cast<float>(man) * 0.001953125f));
  return __uint_as_float(sign | ((ex + 120u) << 23) | (man << 20));
}

// ---------------------------------------------------------------------------
// E2M1 (OCP MX: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign).
// Encoder: nearest grid value, ties to the even code, saturate at 6, NaN -> 6.
// Each comparison counts one grid midpoint passed; strict for midpoints whose
// lower neighbour has the even code, non-strict where the upper one has it.
__device__ __forceinline__ uint32_t e2m1_encode(float y) {
  const uint32_t sign = (__float_as_uint(y) >> 28) & 0x8u;
  const float a = fabsf(y);
  if (a != a) return 0x7u | sign;
  const uint32_t code = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                        (a >= 3.5f) + (a > 5.0f);
  return code | sign;
}

__device__ __forceinline__ float e2m1_decode(uint32_t c) {
  // magnitude bits as a tiny float: code k -> {0, .5, 1, 1.5, 2, 3, 4, 6}
  const uint32_t k = c & 0x7u;
  const float mag = (k < 2u) ? 0.5f * static_cast<float>(k)
                             : __uint_as_float(((126u + (k >> 1)) << 23) | ((k & 1u) << 22));
  return (c & 0x8u) ? -mag : mag;
}

// ---------------------------------------------------------------------------
// Cache geometry.
__host__ __device__ __forceinline__ int64_t page_bytes_of(int kv_dtype, int bs, int hkv, int d) {
  const int64_t elems = static_cast<int64_t>(bs) * hkv * d;
  if (kv_dtype == PD_KV_BF16) return elems * 2;
  if (kv_dtype == PD_KV_FP8_E4M3) return elems;
  return (elems / 2 + elems / 16 + 127) / 128 * 128;
}
__host__ __device__ __forceinline__ int64_t nvfp4_data_bytes(int bs, int hkv, int d) {
  return static_cast<int64_t>(bs) * hkv * d / 2;
}

// ---------------------------------------------------------------------------
// Split geometry. Keys of sequence b are j in [lo, L): lo = L - W when a
// window W > 0 is shorter than L, else 0. They occupy the pages
// lo/bs .. (L-1)/bs of the sequence's block-table row. Every split owns
// `chunk` consecutive pages of that range (the last may be shorter), so the
// first ceil(P_b / chunk) splits of a sequence hold keys and the rest none.
// chunk = ceil(span / S) with span the most pages any sequence can touch.
__host__ __device__ __forceinline__ int window_lo(int L, int W) {
  return (W > 0 && L > W) ? L - W : 0;
}
__host__ __device__ __forceinline__ int num_key_pages(int L, int W, int bs) {
  const int lo = window_lo(L, W);
  return L > lo ? (L - 1) / bs - lo / bs + 1 : 0;
}
__host__ __device__ __forceinline__ int page_span_max(int mbs, int bs, int W) {
  if (W <= 0) return mbs;
  const int span = (W + bs - 1) / bs + 1;
  return span < mbs ? span : mbs;
}
__host__ __device__ __forceinline__ int chunk_pages(int span, int S) {
  const int c = (span + S - 1) / S;
  return c > 0 ? c : 1;
}

// Workspace: O [B][Hq][S][D] fp32, then ML [B][Hq][S] (m, l) fp32 pairs,
// each region starting on a 256-byte boundary.
__host__ __device__ __forceinline__ size_t ws_o_bytes(int B, int Hq, int D, int S) {
  return (static_cast<size_t>(B) * Hq * S * D * sizeof(float) + 255) / 256 * 256;
}
__host__ __device__ __forceinline__ size_t ws_ml_bytes(int B, int Hq, int S) {
  return (static_cast<size_t>(B) * Hq * S * 2 * sizeof(float) + 255) / 256 * 256;
}
__host__ __device__ __forceinline__ size_t ws_total_bytes(int B, int Hq, int D, int S) {
  return ws_o_bytes(B, Hq, D, S) + ws_ml_bytes(B, Hq, S);
}

// ---------------------------------------------------------------------------
// Kernel argument blocks.
struct DecodeArgs {
  const uint16_t* q;             // [B][Hq][D] bf16, sequence b's rows at b * q_stride
  int64_t q_stride;              // elements between consecutive sequences' q rows
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;   // [B][MBS]
  const int32_t* seq_lens;       // [B]
  float* ws_o;                   // [B][Hq][S][D]
  float2* ws_ml;                 // [B][Hq][S]
  int* flags;                    // device status word
  uint16_t* out;                 // [B][Hq][D] bf16 output (used when direct != 0),
                                 // sequence b's rows at b * out_stride
  int64_t out_stride;            // elements between consecutive sequences' output rows
  int direct;                    // 1: a sequence whose keys fit one split writes out
                                 // itself (and an empty one zero rows); the combine
                                 // then skips those sequences
  int64_t num_blocks;
  int64_t page_bytes;
  int64_t data_bytes;            // NVFP4 data-section bytes
  int num_seqs, num_q_heads, num_kv_heads, group, block_size, max_blocks_per_seq;
  int num_splits, chunk, sliding_window;
  // balanced plan (pd_decode_balanced only): per-CTA piece ranges and the
  // pieces (sequence * Hkv + kv head, first key, end key, flags)
  const int32_t* plan_cta;
  const int4* plan_pieces;
  int plan_num_ctas, plan_num_pieces;
  float scale_log2;              // scale * log2(e)
  float k_scale, v_scale;
  // limit of the consumer warps' waits for a stage of keys (ns; ~2 s unless a
  // test shortens it to make the waits run out)
  uint32_t consumer_wait_ns;
};

struct CombineArgs {
  const float* ws_o;
  const float2* ws_ml;
  const int32_t* seq_lens;
  uint16_t* out;                 // sequence b's rows at b * out_stride
  int64_t out_stride;
  int num_seqs, num_q_heads, block_size, max_blocks_per_seq, num_splits, chunk, sliding_window;
  int skip_direct;               // 1: sequences with one key-holding split are already written
  // balanced plan: per (sequence, kv head) its first piece and piece count;
  // when set, the partials of q head h are pieces first.. of its kv head
  // (row piece * group + h % group) instead of the S splits
  const int32_t* plan_seg;
  int num_kv_heads;
  // E4M3 output (pd_decode_e4m3_out): when out8 is set, the combine writes
  // E4M3(o / out_scale) bytes there (row b at b * out_stride) instead of bf16
  uint8_t* out8;
  float out_scale;
};

// Paged prefill: sequence b's query rows are cu_q[b] .. cu_q[b+1]-1 of q and
// out (row r at r * q_stride / r * out_stride elements, Hq * D values each).
struct PrefillArgs {
  const uint16_t* q;
  int64_t q_stride;
  const int32_t* cu_q;           // [B + 1]
  const int32_t* block_tables;   // [B][MBS]
  const int32_t* seq_lens;       // [B], keys in the cache, the new tokens included
  uint16_t* out;
  int64_t out_stride;
  int* flags;
  int64_t num_blocks;
  int num_seqs, num_q_heads, num_kv_heads, group, block_size, max_blocks_per_seq;
  int tokens_per_cta;            // query tokens of one CTA: 64 / group
  int causal, sliding_window;
  float scale_log2;              // scale * log2(e)
  const void* k_cache;           // the caches (read by bulk copies for NVFP4)
  const void* v_cache;
  float k_scale, v_scale;        // FP8 per-tensor scales
};

// Sequence length as the kernels use it: clamped to the block table, with a
// flag raised for values outside [0, MBS*bs].
__device__ __forceinline__ int checked_seq_len(const int32_t* seq_lens, int b, int mbs, int bs,
                                               int* flags) {
  int L = seq_lens[b];
  const int cap = mbs * bs;
  if (L < 0 || L > cap) {
    atomicOr(flags, PD_DEV_BAD_SEQ_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

}  // namespace pd

// Launchers (defined in the kernel translation units).
namespace pd {
// pd_decode's argument checks, in the order it reports them, up to (not
// including) the workspace; a split count of 0 is resolved to the automatic
// choice on the current device. Defined in pd_api.cu; pd_decode_static_ws
// uses it so that both calls answer a malformed request with the same code.
int decode_checks(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* seq_lens, const void* out,
                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                  int32_t num_splits, int32_t sliding_window, int32_t kv_dtype, float k_scale,
                  float v_scale, int64_t q_stride, int64_t out_stride, int* num_splits_out);
cudaError_t launch_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint8_t* kc,
                                     uint8_t* vc, const int32_t* slots, int T, int hkv, int d,
                                     int bs, int64_t nb, int kv_dtype, float k_scale,
                                     float v_scale, int* flags, cudaStream_t st);
cudaError_t launch_absmax(const uint16_t* data, int64_t n, float* out, int num_sms,
                          cudaStream_t st);
cudaError_t launch_fp8_scales(const float* absmax, float* scales, int n, cudaStream_t st);
// The cache write's E4M3 (format 0) / E2M1 (format 1) encoders on the fp32 bit
// patterns first .. first + n - 1 (wrapping), one code byte each (a test hook).
cudaError_t launch_encode_bits(int format, uint32_t first, int64_t n, uint8_t* out, int num_sms,
                               cudaStream_t st);
cudaError_t launch_decode_partial(const DecodeArgs& a, int head_dim, int kv_dtype,
                                  cudaStream_t st);
cudaError_t launch_decode_partial_mma(const DecodeArgs& a, int head_dim, int kv_dtype,
                                      cudaStream_t st);
// Resident CTAs per SM of the tensor-core partial kernel, from its shared
// memory per CTA (host-only estimate; no CUDA call).
int mma_ctas_per_sm_estimate(int kv_dtype, int head_dim);
cudaError_t launch_decode_partial_balanced(const DecodeArgs& a, int head_dim, int kv_dtype,
                                           cudaStream_t st);
// Resident CTAs per SM of the balanced partial kernel for a GQA group size.
int balanced_ctas_per_sm(int kv_dtype, int head_dim, int group);
// max_parts: the most partials any row has (sizes the combine's CTAs)
cudaError_t launch_decode_combine(const CombineArgs& a, int head_dim, int max_parts,
                                  cudaStream_t st);
// Paged prefill (head_dim 64 / 128 / 256).
// launch_prefill: mma.sync kernel, any cache form, 64 rows per CTA
// (tokens_per_cta = 64 / G); launch_prefill_pair: tcgen05 kernel, BF16
// caches, head_dim 64 / 128, two 128-row query tiles per CTA
// (tokens_per_cta = 128 / G per tile); launch_prefill_umma: tcgen05 kernel,
// BF16 caches, head_dim 256, one 128-row tile per CTA (128 / G).
cudaError_t launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                           int head_dim, int kv_dtype, int max_q_len, cudaStream_t st);
cudaError_t launch_prefill_pair(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                                int head_dim, int max_q_len, cudaStream_t st);
cudaError_t launch_prefill_umma(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                                int head_dim, int max_q_len, cudaStream_t st);
}  // namespace pd
