/*
 * Plain CPU oracle for paged split-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library. The product
 * path (paged_kv_split_gb300 and libpd.so) never calls it and shares no code,
 * header, table or helper with it.
 *
 * Plain C++17, single-threaded, fp32 arithmetic, built with -O2
 * -ffp-contract=off and without -ffast-math, so every rounding step below is
 * the IEEE fp32 operation written in the source.
 *
 * What it computes follows three pages:
 *   - metrale, "prefill_attn_b.rs" (launchers `reshape_and_cache_nvfp4`,
 *     `bf16_absmax`, `paged_decode_attn_splitk_{nvfp4,fp8,bf16}`,
 *     `paged_decode_attn_reduce_{nvfp4,fp8}`): the cache formats (BF16 cache
 *     `[blocks, block_size, kv_heads, head_dim]`; FP8 E4M3 with per-tensor
 *     k_scale / v_scale; NVFP4 = E2M1 values with one E4M3 scale per 16, a
 *     data section followed by scales inside a page of `block_stride_bytes`),
 *     the block table `[num_seqs, max_blocks_per_seq]`, `slot_mapping`,
 *     `seq_lens`, `sliding_window`, `inv_sqrt_d`.
 *   - AstrAI, "csrc/tests" commit log: int32 page-table and cache-location
 *     indices, the scale applied after the dot product, fmaf() for the V
 *     accumulation, expf for the exponent, 1e-20 divide-by-zero guards.
 *   - pegainfer issue 1008: the decode / split-KV decode units over a paged KV
 *     view.
 *
 * Decode attention reaches the plain softmax attention result exactly (up to
 * rounding order), so oracle_decode is that definition written out token by
 * token through the block table: two-pass softmax, no splits, no tiling.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - E4M3 / E2M1 encoders round to nearest, ties to even mantissa, and
 *     saturate finite overflow and +-Inf to the largest finite magnitude
 *     (448 / 6). The sign of a value that rounds to zero is kept.
 *     E4M3 NaN input -> 0x7F | sign; E2M1 has no NaN, so NaN saturates to 6.
 *   - FP8 quantisation divides: code = E4M3(float(x) / scale); a NaN input
 *     keeps its own sign (IEEE does not fix the sign of a NaN quotient).
 *   - FP8 calibration scale = amax / 448 (1.0 when amax == 0).
 *   - NVFP4 group scale = E4M3(amax / 6), amax over the 16 values with NaN
 *     skipped; a group whose decoded scale is 0 stores +0 codes; otherwise
 *     code_i = E2M1(float(x_i) / scale).
 *   - NVFP4 page = data section [kv_heads][block_size][head_dim/2] (element
 *     2i in the low nibble, 2i+1 in the high nibble), then the scale section
 *     [kv_heads][block_size][head_dim/16], page padded to a multiple of 128 B.
 *   - slot = page * block_size + offset; a negative slot skips the token.
 *   - Sliding window W > 0 keeps keys j with (L-1) - j < W; W = 0 is off.
 *   - GQA: q head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - A sequence with no key in range produces a zero output row.
 *   - Output = fp32 -> bf16 round to nearest even.
 */
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

constexpr int KV_BF16 = 0;
constexpr int KV_FP8 = 1;
constexpr int KV_NVFP4 = 2;

float bits_to_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
uint32_t float_to_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

/* bfloat16 is the top half of an IEEE binary32. */
float bf16_value(uint16_t b) { return bits_to_float(static_cast<uint32_t>(b) << 16); }

/* Round a binary32 to the nearest bfloat16, ties to even; NaN stays NaN. */
uint16_t bf16_round(float f) {
  uint32_t u = float_to_bits(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return static_cast<uint16_t>(upper);
}

/* Round a non-negative value that is an exact multiple of a power of two
 * away from an integer to the nearest integer, ties to even. */
double round_half_even(double y) {
  double fl = std::floor(y);
  double frac = y - fl;
  if (frac > 0.5) return fl + 1.0;
  if (frac < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* ---- OCP E4M3 ("E4M3FN"): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, largest finite 448 (S.1111.110),
 * subnormals m/8 * 2^-6. */
float e4m3_value(uint8_t c) {
  const int sign = c >> 7;
  const int ex = (c >> 3) & 0xF;
  const int man = c & 0x7;
  float mag;
  if (ex == 0xF && man == 0x7) {
    mag = std::numeric_limits<float>::quiet_NaN();
  } else if (ex == 0) {
    mag = std::ldexp(static_cast<float>(man) / 8.0f, -6);
  } else {
    mag = std::ldexp(1.0f + static_cast<float>(man) / 8.0f, ex - 7);
  }
  return sign ? -mag : mag;
}

uint8_t e4m3_code(float x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return static_cast<uint8_t>(0x7F | sign);
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return static_cast<uint8_t>(0x7E | sign); /* saturate (incl. Inf) */
  if (a < std::ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9; n == 8 is the smallest normal 2^-6,
     * whose code is 8 as well. */
    const double n = round_half_even(a * 512.0);
    return static_cast<uint8_t>(static_cast<int>(n) | sign);
  }
  int e2;
  std::frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;              /* a in [2^e, 2^(e+1)) */
  double n = round_half_even(std::ldexp(a, 3 - e)); /* in [8, 16] */
  if (n == 16.0) {
    e += 1;
    n = 8.0;
  }
  const int field = e + 7;
  const int man = static_cast<int>(n) - 8;
  if (field > 15 || (field == 15 && man == 7)) return static_cast<uint8_t>(0x7E | sign);
  return static_cast<uint8_t>(((field << 3) | man) | sign);
}

/* ---- OCP E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no
 * Inf / NaN, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}. Codes are 4 bits. */
float e2m1_value(uint8_t c) {
  const int sign = (c >> 3) & 1;
  const int ex = (c >> 1) & 0x3;
  const int man = c & 0x1;
  float mag;
  if (ex == 0) {
    mag = 0.5f * static_cast<float>(man);
  } else {
    mag = std::ldexp(1.0f + 0.5f * static_cast<float>(man), ex - 1);
  }
  return sign ? -mag : mag;
}

uint8_t e2m1_code(float x) {
  const uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  if (std::isnan(x)) return static_cast<uint8_t>(0x7 | sign);
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 6.0) return static_cast<uint8_t>(0x7 | sign);
  if (a < 1.0) {
    const double n = round_half_even(a * 2.0); /* quantum 0.5; n == 2 is 1.0 = code 2 */
    return static_cast<uint8_t>(static_cast<int>(n) | sign);
  }
  int e2;
  std::frexp(a, &e2);
  int e = e2 - 1;                                    /* a in [2^e, 2^(e+1)), e in {0,1,2} */
  double n = round_half_even(std::ldexp(a, 1 - e)); /* in [2, 4] */
  if (n == 4.0) {
    e += 1;
    n = 2.0;
  }
  const int field = e + 1;
  const int man = static_cast<int>(n) - 2;
  if (field > 3) return static_cast<uint8_t>(0x7 | sign);
  return static_cast<uint8_t>(((field << 1) | man) | sign);
}

/* x / s in IEEE fp32; a NaN x is passed through unchanged so that its sign
 * (which IEEE leaves unspecified for a NaN quotient) selects the code. */
float quotient(float x, float s) { return std::isnan(x) ? x : x / s; }

/* ---- Cache geometry (bytes). */
int64_t page_bytes(int kv_dtype, int32_t bs, int32_t hkv, int32_t d) {
  const int64_t elems = static_cast<int64_t>(bs) * hkv * d;
  if (kv_dtype == KV_BF16) return elems * 2;
  if (kv_dtype == KV_FP8) return elems;
  const int64_t raw = elems / 2 + elems / 16;
  return (raw + 127) / 128 * 128;
}
int64_t nvfp4_data_bytes(int32_t bs, int32_t hkv, int32_t d) {
  return static_cast<int64_t>(bs) * hkv * d / 2;
}

/* Dequantised row of one (page, row-in-page, kv head) of a cache, fp32. */
void read_row(const uint8_t* cache, int kv_dtype, int64_t page, int32_t off, int32_t head,
              int32_t bs, int32_t hkv, int32_t d, float scale, float* row) {
  const int64_t pb = page_bytes(kv_dtype, bs, hkv, d);
  const uint8_t* base = cache + page * pb;
  if (kv_dtype == KV_BF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base) +
                        (static_cast<int64_t>(off) * hkv + head) * d;
    for (int32_t i = 0; i < d; ++i) row[i] = bf16_value(p[i]);
  } else if (kv_dtype == KV_FP8) {
    const uint8_t* p = base + (static_cast<int64_t>(off) * hkv + head) * d;
    for (int32_t i = 0; i < d; ++i) row[i] = e4m3_value(p[i]) * scale;
  } else {
    const uint8_t* data = base + (static_cast<int64_t>(head) * bs + off) * (d / 2);
    const uint8_t* sc = base + nvfp4_data_bytes(bs, hkv, d) +
                        (static_cast<int64_t>(head) * bs + off) * (d / 16);
    for (int32_t i = 0; i < d; ++i) {
      const uint8_t byte = data[i / 2];
      const uint8_t code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      row[i] = e2m1_value(code) * e4m3_value(sc[i / 16]);
    }
  }
}

/* One query vector qh (q head h, kv head h / group) over keys [lo, hi) of
 * sequence b, straight from the definition: scores s_j = scale * sum_d
 * q[d] * k_j[d] (fp32, scale after the dot), two-pass softmax with expf,
 * out = sum_j e_j v_j (fmaf) / max(sum_j e_j, 1e-20), then bf16. An empty
 * range gives a zero row. Writes oh (bf16) and, if not null, of (fp32);
 * returns false for an out-of-range page index. */
bool attend_one(const uint16_t* qh, int32_t h, int32_t group, int32_t b, int32_t lo, int32_t hi,
                const uint8_t* k_cache, const uint8_t* v_cache, const int32_t* block_tables,
                int32_t max_blocks_per_seq, int64_t num_blocks, int32_t num_kv_heads,
                int32_t head_dim, int32_t block_size, float scale, int32_t kv_dtype,
                float k_scale, float v_scale, uint16_t* oh, float* of) {
  const int32_t g = h / group;
  const int32_t n = hi > lo ? hi - lo : 0;
  std::vector<float> krow(head_dim), vrow(head_dim), acc(head_dim, 0.0f), s(n);
  for (int32_t j = lo; j < hi; ++j) {
    const int64_t page = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + j / block_size];
    if (page < 0 || page >= num_blocks) return false;
    read_row(k_cache, kv_dtype, page, j % block_size, g, block_size, num_kv_heads, head_dim,
             k_scale, krow.data());
    float dot = 0.0f;
    for (int32_t i = 0; i < head_dim; ++i) dot = dot + bf16_value(qh[i]) * krow[i];
    s[j - lo] = scale * dot;
  }
  float m = -std::numeric_limits<float>::infinity();
  for (int32_t j = 0; j < n; ++j)
    if (s[j] > m) m = s[j];
  float l = 0.0f;
  for (int32_t j = 0; j < n; ++j) {
    s[j] = std::exp(s[j] - m);
    l = l + s[j];
  }
  for (int32_t j = lo; j < hi; ++j) {
    const int64_t page = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + j / block_size];
    read_row(v_cache, kv_dtype, page, j % block_size, g, block_size, num_kv_heads, head_dim,
             v_scale, vrow.data());
    const float e = s[j - lo];
    for (int32_t i = 0; i < head_dim; ++i) acc[i] = std::fmaf(e, vrow[i], acc[i]);
  }
  const float denom = l > 1e-20f ? l : 1e-20f;
  for (int32_t i = 0; i < head_dim; ++i) {
    const float o = acc[i] / denom;
    oh[i] = bf16_round(o);
    if (of) of[i] = o;
  }
  return true;
}

}  // namespace

extern "C" {

/* Codec entry points, exported so tests can pin them directly. */
float oracle_bf16_value(uint16_t b) { return bf16_value(b); }
uint16_t oracle_bf16_round(float f) { return bf16_round(f); }
float oracle_e4m3_value(uint8_t c) { return e4m3_value(c); }
uint8_t oracle_e4m3_code(float x) { return e4m3_code(x); }
float oracle_e2m1_value(uint8_t c) { return e2m1_value(c); }
uint8_t oracle_e2m1_code(float x) { return e2m1_code(x); }

void oracle_e4m3_code_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(x[i]);
}
void oracle_e2m1_code_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_code(x[i]);
}

int64_t oracle_page_bytes(int32_t kv_dtype, int32_t block_size, int32_t num_kv_heads,
                          int32_t head_dim) {
  return page_bytes(kv_dtype, block_size, num_kv_heads, head_dim);
}

/* max |x| over n bf16 values; NaN values are skipped (metrale `bf16_absmax`). */
float oracle_absmax_bf16(const uint16_t* data, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    const float a = std::fabs(bf16_value(data[i]));
    if (a > m) m = a;
  }
  return m;
}

/* FP8 per-tensor scale from the calibration absmax: amax / 448 (1 if 0). */
float oracle_fp8_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

/* Write each token's K and V rows into the paged cache at slot_mapping[t]
 * (metrale `reshape_and_cache_nvfp4`, extended to the BF16 and FP8 forms).
 * key / value: bf16 [num_tokens, num_kv_heads, head_dim], contiguous.
 * Returns 0, or -1 for an out-of-range slot or a bad shape. */
int oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint8_t* k_cache,
                             uint8_t* v_cache, const int32_t* slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, int32_t kv_dtype, float k_scale, float v_scale) {
  if (kv_dtype == KV_NVFP4 && head_dim % 16 != 0) return -1;
  const int64_t pb = page_bytes(kv_dtype, block_size, num_kv_heads, head_dim);
  for (int32_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * block_size) return -1;
    const int64_t page = slot / block_size;
    const int32_t off = static_cast<int32_t>(slot % block_size);
    for (int which = 0; which < 2; ++which) {
      const uint16_t* src = (which == 0 ? key : value) +
                            static_cast<int64_t>(t) * num_kv_heads * head_dim;
      uint8_t* cache = (which == 0 ? k_cache : v_cache);
      const float sc = (which == 0 ? k_scale : v_scale);
      uint8_t* base = cache + page * pb;
      for (int32_t h = 0; h < num_kv_heads; ++h) {
        const uint16_t* x = src + static_cast<int64_t>(h) * head_dim;
        if (kv_dtype == KV_BF16) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(base) +
                          (static_cast<int64_t>(off) * num_kv_heads + h) * head_dim;
          for (int32_t i = 0; i < head_dim; ++i) dst[i] = x[i];
        } else if (kv_dtype == KV_FP8) {
          uint8_t* dst = base + (static_cast<int64_t>(off) * num_kv_heads + h) * head_dim;
          for (int32_t i = 0; i < head_dim; ++i) dst[i] = e4m3_code(quotient(bf16_value(x[i]), sc));
        } else {
          uint8_t* data = base + (static_cast<int64_t>(h) * block_size + off) * (head_dim / 2);
          uint8_t* scl = base + nvfp4_data_bytes(block_size, num_kv_heads, head_dim) +
                         (static_cast<int64_t>(h) * block_size + off) * (head_dim / 16);
          for (int32_t g = 0; g < head_dim / 16; ++g) {
            float amax = 0.0f;
            for (int32_t i = 0; i < 16; ++i) {
              const float a = std::fabs(bf16_value(x[g * 16 + i]));
              if (a > amax) amax = a; /* NaN compares false: skipped */
            }
            const uint8_t scode = e4m3_code(amax / 6.0f);
            const float s = e4m3_value(scode);
            scl[g] = scode;
            for (int32_t i = 0; i < 16; i += 2) {
              uint8_t lo = 0, hi = 0;
              if (s != 0.0f) {
                lo = e2m1_code(quotient(bf16_value(x[g * 16 + i]), s));
                hi = e2m1_code(quotient(bf16_value(x[g * 16 + i + 1]), s));
              }
              data[(g * 16 + i) / 2] = static_cast<uint8_t>(lo | (hi << 4));
            }
          }
        }
      }
    }
  }
  return 0;
}

/* Decode attention for every (sequence, q head), straight from the
 * definition: scores s_j = scale * sum_d q[d] * k_j[d] over the keys in the
 * window, two-pass softmax, out = sum_j e_j v_j / sum_j e_j, then bf16.
 * q: bf16 [num_seqs, num_q_heads, head_dim]; out: bf16 of the same shape;
 * out_f32 (may be null) receives the value before the bf16 rounding.
 * Returns 0, or -1 for a bad shape or an out-of-range page index. */
int oracle_decode(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                  const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out,
                  float* out_f32, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                  int64_t num_blocks, float scale, int32_t sliding_window, int32_t kv_dtype,
                  float k_scale, float v_scale) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
  if (kv_dtype == KV_NVFP4 && head_dim % 16 != 0) return -1;
  const int32_t group = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t len = seq_lens[b];
    if (len < 0 || static_cast<int64_t>(len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
      return -1;
    const int32_t lo = (sliding_window > 0 && len > sliding_window) ? len - sliding_window : 0;
    for (int32_t h = 0; h < num_q_heads; ++h) {
      const int64_t row = static_cast<int64_t>(b) * num_q_heads + h;
      if (!attend_one(q + row * head_dim, h, group, b, lo, len, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, num_blocks, num_kv_heads, head_dim, block_size, scale,
                      kv_dtype, k_scale, v_scale, out + row * head_dim,
                      out_f32 ? out_f32 + row * head_dim : nullptr))
        return -1;
    }
  }
  return 0;
}

/* Decode with E4M3 output codes (the "E4M3 output variant" the AstrAI
 * "csrc/tests" log names beside stride-based addressing, which the pages do
 * not define further). Reading taken: out_codes[b, h, d] =
 * E4M3(o[b, h, d] / out_scale), where o is the fp32 attention output that
 * oracle_decode computes before its bf16 rounding, out_scale a per-tensor
 * fp32 scale (finite, > 0), the division IEEE fp32, and the encoder the
 * cache's (nearest, ties to even, saturation to +-448, sign of zero kept).
 * The stored code decodes to code * out_scale. Returns 0, or -1 as
 * oracle_decode (or for a bad out_scale). */
int oracle_decode_e4m3_out(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           uint8_t* out_codes, int32_t num_seqs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                           int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                           float out_scale) {
  if (!(std::isfinite(out_scale) && out_scale > 0.0f)) return -1;
  const size_t n = static_cast<size_t>(num_seqs) * num_q_heads * head_dim;
  std::vector<uint16_t> out_bf16(n);
  std::vector<float> o(n);
  const int rc = oracle_decode(q, k_cache, v_cache, block_tables, seq_lens, out_bf16.data(),
                               o.data(), num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, max_blocks_per_seq, num_blocks, scale,
                               sliding_window, kv_dtype, k_scale, v_scale);
  if (rc != 0) return rc;
  for (size_t i = 0; i < n; ++i) out_codes[i] = e4m3_code(quotient(o[i], out_scale));
  return 0;
}

/* Paged prefill (chunked prefill) attention over the same caches: several
 * query tokens per sequence. The pages name this unit beside decode
 * (pegainfer issue 1008: `prefill_paged_launch` over the paged-KV view;
 * AstrAI "csrc/tests" log: prefill kernels templated on the paged KV source,
 * one `causal_offset` with -1 = off and >= 0 = the first query position,
 * stride addressing for Q/KV/O). Sequence b owns query rows
 * [cu_q[b], cu_q[b+1]) of q and out (bf16 [total_q, num_q_heads, head_dim])
 * and L_b = seq_lens[b] keys in the cache, its new tokens included, so
 * q_len_b <= L_b. causal != 0: the queries are the sequence's newest tokens,
 * query i at position p = L_b - q_len_b + i, and it sees keys j <= p (the
 * first query position of sequence b is L_b - q_len_b). causal == 0: every
 * query sees all L_b keys, p = L_b - 1. A window W > 0 keeps keys j with
 * p - j < W. Each (query, head) is then the decode definition above over
 * keys [lo, p + 1): fp32 dot, scale after the dot, two-pass softmax with
 * expf, fmaf accumulation of V, 1e-20 guard, bf16 round to nearest even.
 * Returns 0, or -1 for a bad shape or an out-of-range page index. */
int oracle_prefill(const uint16_t* q, const int32_t* cu_q, const uint8_t* k_cache,
                   const uint8_t* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                   uint16_t* out, float* out_f32, int32_t num_seqs, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t causal,
                   int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
  if (kv_dtype == KV_NVFP4 && head_dim % 16 != 0) return -1;
  const int32_t group = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t len = seq_lens[b];
    const int32_t q_len = cu_q[b + 1] - cu_q[b];
    if (len < 0 || q_len < 0 || q_len > len ||
        static_cast<int64_t>(len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
      return -1;
    for (int32_t i = 0; i < q_len; ++i) {
      const int64_t qrow = static_cast<int64_t>(cu_q[b]) + i;
      const int32_t pos = causal ? len - q_len + i : len - 1;  // the query's position
      const int32_t hi = pos + 1;                               // keys [lo, hi)
      const int32_t lo = (sliding_window > 0 && hi > sliding_window) ? hi - sliding_window : 0;
      for (int32_t h = 0; h < num_q_heads; ++h) {
        const int64_t row = qrow * num_q_heads + h;
        if (!attend_one(q + row * head_dim, h, group, b, lo, hi, k_cache, v_cache, block_tables,
                        max_blocks_per_seq, num_blocks, num_kv_heads, head_dim, block_size, scale,
                        kv_dtype, k_scale, v_scale, out + row * head_dim,
                        out_f32 ? out_f32 + row * head_dim : nullptr))
          return -1;
      }
    }
  }
  return 0;
}

}  // extern "C"
