// Split-KV partial (CUDA-core form) and the log-sum-exp combine.
//
// metrale "prefill_attn_b.rs": `paged_decode_attn_splitk_{nvfp4,fp8,bf16}` cut
// each sequence's keys into num_splits parts, each block writing its partial
// output and softmax state (F32 [head_dim values, m, l]) to a workspace, and
// `paged_decode_attn_reduce_*` combine them into the BF16 output, reading
// seq_lens. AstrAI "csrc/tests": split-KV decode with o_part / ml_part and a
// single combine kernel; fmaf for the V accumulation; 1e-20 divide guards.
//
// This partial kernel is the plain form: one CTA per (sequence, kv head,
// split) packs the whole GQA group so every K/V element is read once per kv
// head; scores use warp reductions over head_dim; online softmax over tiles
// of 64 keys; V accumulation in fp32 registers. Scores are kept in log2
// units (scale * log2(e) folded into q), exponentials are exp2f.
#include "pd_common.cuh"

namespace pd {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 64;

// Dequantised element d of the (page, row, head) row of a cache.
template <int FMT>
__device__ __forceinline__ float load_kv(const uint8_t* __restrict__ cache, int64_t page, int row,
                                         int head, int d, const DecodeArgs& a, int D, float sc) {
  const uint8_t* base = cache + page * a.page_bytes;
  if (FMT == PD_KV_BF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base) +
                        (static_cast<int64_t>(row) * a.num_kv_heads + head) * D + d;
    return bf16_to_f32(*p);
  } else if (FMT == PD_KV_FP8_E4M3) {
    const uint8_t* p = base + (static_cast<int64_t>(row) * a.num_kv_heads + head) * D + d;
    return e4m3_decode(*p) * sc;
  } else {
    const int64_t line = static_cast<int64_t>(head) * a.block_size + row;
    const uint8_t byte = base[line * (D / 2) + d / 2];
    const uint32_t code = (d & 1) ? (byte >> 4) : (byte & 0xFu);
    const float s = e4m3_decode(base[a.data_bytes + line * (D / 16) + d / 16]);
    return e2m1_decode(code) * s;
  }
}

template <int FMT, int D>
__global__ void __launch_bounds__(kThreads) partial_simple_kernel(const DecodeArgs a) {
  // let the dependent combine grid be scheduled as this grid drains
  asm volatile("griddepcontrol.launch_dependents;");
  // Launched as a programmatic dependent of whatever came before on the
  // stream (the previous step's combine, say): nothing global is read or
  // written before that grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kPerLane = D / 32;
  constexpr int kAccMax = kMaxGroup * D / kThreads;
  const int g = blockIdx.x;  // kv head
  const int s = blockIdx.y;  // split
  const int b = blockIdx.z;  // sequence
  const int G = a.group;
  const int bs = a.block_size;
  const int L = checked_seq_len(a.seq_lens, b, a.max_blocks_per_seq, bs, a.flags);
  const int lo = window_lo(L, a.sliding_window);
  const int P = num_key_pages(L, a.sliding_window, bs);
  if (s * a.chunk >= P) return;  // this split holds no key of sequence b
  const int first_page = lo / bs + s * a.chunk;
  const int last_page = min(lo / bs + P, first_page + a.chunk);  // exclusive
  const int t_begin = max(lo, first_page * bs);
  const int t_end = min(L, last_page * bs);

  extern __shared__ float smem[];
  float* qs = smem;                 // [G][D], q * scale * log2(e)
  float* sc = qs + G * D;           // [G][kTile] scores, then probabilities
  float* m_s = sc + G * kTile;      // [G] running max (log2 units)
  float* l_s = m_s + kMaxGroup;     // [G] running sum
  float* alpha_s = l_s + kMaxGroup; // [G] rescale factor of the current tile

  const uint16_t* qg = a.q + static_cast<int64_t>(b) * a.q_stride + g * G * D;
  for (int i = threadIdx.x; i < G * D; i += kThreads) qs[i] = bf16_to_f32(qg[i]) * a.scale_log2;
  if (threadIdx.x < G) {
    m_s[threadIdx.x] = -INFINITY;
    l_s[threadIdx.x] = 0.0f;
  }
  float acc[kAccMax];
#pragma unroll
  for (int k = 0; k < kAccMax; ++k) acc[k] = 0.0f;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

  for (int t0 = t_begin; t0 < t_end; t0 += kTile) {
    const int n = min(kTile, t_end - t0);
    // scores: one warp per key, lanes over head_dim
    for (int tt = warp; tt < n; tt += kWarps) {
      const int j = t0 + tt;
      const int64_t page = bt[j / bs];
      const bool ok = page >= 0 && page < a.num_blocks;
      float kv[kPerLane];
#pragma unroll
      for (int i = 0; i < kPerLane; ++i)
        kv[i] = ok ? load_kv<FMT>(a.k_cache, page, j % bs, g, lane + 32 * i, a, D, a.k_scale)
                   : 0.0f;
      for (int h = 0; h < G; ++h) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) part = fmaf(qs[h * D + lane + 32 * i], kv[i], part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        if (lane == 0) sc[h * kTile + tt] = ok ? part : -INFINITY;
      }
      if (!ok && lane == 0) atomicOr(a.flags, PD_DEV_BAD_PAGE);
    }
    __syncthreads();
    // online softmax update, one thread per q head
    if (threadIdx.x < G) {
      const int h = threadIdx.x;
      float mx = m_s[h];
      for (int tt = 0; tt < n; ++tt) mx = fmaxf(mx, sc[h * kTile + tt]);
      const float alpha = (mx == -INFINITY) ? 1.0f : exp2f(m_s[h] - mx);
      float l = l_s[h] * alpha;
      for (int tt = 0; tt < n; ++tt) {
        const float p = (mx == -INFINITY) ? 0.0f : exp2f(sc[h * kTile + tt] - mx);
        sc[h * kTile + tt] = p;
        l += p;
      }
      m_s[h] = mx;
      l_s[h] = l;
      alpha_s[h] = alpha;
    }
    __syncthreads();
    // acc[h][d] = alpha * acc + sum_t p[h][t] * v_t[d]
#pragma unroll
    for (int k = 0; k < kAccMax; ++k) {
      const int e = threadIdx.x + k * kThreads;
      if (e < G * D) {
        const int h = e / D;
        const int d = e % D;
        float v = acc[k] * alpha_s[h];
        for (int tt = 0; tt < n; ++tt) {
          const int j = t0 + tt;
          const int64_t page = bt[j / bs];
          if (page < 0 || page >= a.num_blocks) continue;
          const float vv = load_kv<FMT>(a.v_cache, page, j % bs, g, d, a, D, a.v_scale);
          v = fmaf(sc[h * kTile + tt], vv, v);
        }
        acc[k] = v;
      }
    }
    __syncthreads();
  }
  // write the normalised partial and its (m, l)
  const int64_t row0 = (static_cast<int64_t>(b) * a.num_q_heads + g * G) * a.num_splits + s;
#pragma unroll
  for (int k = 0; k < kAccMax; ++k) {
    const int e = threadIdx.x + k * kThreads;
    if (e < G * D) {
      const int h = e / D;
      const int d = e % D;
      const float l = l_s[h];
      a.ws_o[(row0 + static_cast<int64_t>(h) * a.num_splits) * D + d] =
          acc[k] / fmaxf(l, 1e-20f);
    }
  }
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    a.ws_ml[row0 + static_cast<int64_t>(h) * a.num_splits] = make_float2(m_s[h], l_s[h]);
  }
}

// Combine: one CTA per (q head, sequence). D/4 threads span one row (4
// consecutive elements each) and WAYS such lane groups share out the
// partials: group j sums partials j, j + WAYS, ... Each thread's first kRows
// partial rows and their (m, l) are loaded before the weights are found, so
// they all travel together; every warp finds M = max m_s and the weight sum
// by itself with shuffles (no block barrier), and the groups' sums are added
// in group order through shared memory (the one barrier). Weights
// w_s = l_s 2^(m_s - M). The host picks WAYS from the largest partial count
// (one group when a row has only a few partials, as in the balanced
// schedule: small CTAs).
template <int D, int WAYS>
struct CombineShape {
  static constexpr int kLanes = D / 4;          // threads across a row
  static constexpr int kThreads = kLanes * WAYS;
  static constexpr int kRows = 8;               // rows in flight per thread
};

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& o) {
  acc.x = fmaf(w, o.x, acc.x);
  acc.y = fmaf(w, o.y, acc.y);
  acc.z = fmaf(w, o.z, acc.z);
  acc.w = fmaf(w, o.w, acc.w);
}

template <int D, int WAYS, bool E4M3_OUT>
__global__ void __launch_bounds__(CombineShape<D, WAYS>::kThreads)
    combine_kernel(const CombineArgs a) {
  // Launched as a programmatic dependent of the partial kernel: wait until
  // that grid has completed and its workspace writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  using CS = CombineShape<D, WAYS>;
  constexpr int kThreads = CS::kThreads;
  // lanes of the (possibly partial) warp and the first butterfly offset
  constexpr unsigned kMask = kThreads >= 32 ? 0xFFFFFFFFu : ((1u << kThreads) - 1u);
  constexpr int kOff = kThreads >= 32 ? 16 : kThreads / 2;
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  // partial s of this (sequence, q head) is workspace row row0 + s * stride
  int n;
  int64_t row0;
  int stride;
  if (a.plan_seg != nullptr) {
    // balanced plan: the pieces of this q head's kv head, consecutive slots
    const int G = a.num_q_heads / a.num_kv_heads;
    const int g = h / G;
    const int64_t e = 2 * (static_cast<int64_t>(b) * a.num_kv_heads + g);
    n = a.plan_seg[e + 1];
    if (n == 1) return;  // one piece: the partial kernel wrote this row
    row0 = static_cast<int64_t>(a.plan_seg[e]) * G + (h - g * G);
    stride = G;
  } else {
    int L = a.seq_lens[b];
    const int cap = a.max_blocks_per_seq * a.block_size;
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int P = num_key_pages(L, a.sliding_window, a.block_size);
    n = min((P + a.chunk - 1) / a.chunk, a.num_splits);  // splits holding keys
    if (a.skip_direct && n <= 1) return;  // the partial kernel wrote this row
    row0 = (static_cast<int64_t>(b) * a.num_q_heads + h) * a.num_splits;
    stride = 1;
  }
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int j = tid / CS::kLanes;        // partial group (0 .. WAYS-1)
  const int d = (tid % CS::kLanes) * 4;  // first of this thread's 4 elements
  __shared__ __align__(16) float part[WAYS > 1 ? WAYS - 1 : 1][WAYS > 1 ? D : 4];
  const float2* mlp = a.ws_ml + row0;
  const float* op = a.ws_o + row0 * D + d;
  const int64_t ostep = static_cast<int64_t>(stride) * D;  // between consecutive partials
  // this thread's first kRows partial rows and their (m, l), in flight while
  // the weights are found
  float4 o[CS::kRows];
  float2 mlr[CS::kRows];
#pragma unroll
  for (int r = 0; r < CS::kRows; ++r) {
    const int s = j + r * WAYS;
    o[r] = s < n ? *reinterpret_cast<const float4*>(op + s * ostep)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    mlr[r] = s < n ? mlp[s * stride] : make_float2(-INFINITY, 0.0f);
  }
  // every warp finds M = max_s m_s and W = sum_s l_s 2^(m_s - M) by itself
  // (lanes stride over the partials, shuffles combine): no block barrier
  constexpr int kWL = kThreads >= 32 ? 32 : kThreads;  // lanes of a warp
  float M = -INFINITY;
  for (int s = lane; s < n; s += kWL) M = fmaxf(M, mlp[s * stride].x);
#pragma unroll
  for (int off = kOff; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kMask, M, off));
  float wsum = 0.0f;
  if (M != -INFINITY)
    for (int s = lane; s < n; s += kWL) {
      const float2 ml = mlp[s * stride];
      wsum += ml.y * exp2f(ml.x - M);
    }
#pragma unroll
  for (int off = kOff; off > 0; off >>= 1) wsum += __shfl_xor_sync(kMask, wsum, off);
  auto weight = [&](const float2 ml) { return (M == -INFINITY) ? 0.0f : ml.y * exp2f(ml.x - M); };
  // this group's share of sum_s w_s O_s
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < CS::kRows; ++r) {
    const int s = j + r * WAYS;
    if (s < n) fma4(acc, weight(mlr[r]), o[r]);
  }
  for (int s0 = j + CS::kRows * WAYS; s0 < n; s0 += CS::kRows * WAYS) {
#pragma unroll
    for (int r = 0; r < CS::kRows; ++r) {
      const int s = s0 + r * WAYS;
      o[r] = s < n ? *reinterpret_cast<const float4*>(op + s * ostep)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      mlr[r] = s < n ? mlp[s * stride] : make_float2(-INFINITY, 0.0f);
    }
#pragma unroll
    for (int r = 0; r < CS::kRows; ++r) {
      const int s = s0 + r * WAYS;
      if (s < n) fma4(acc, weight(mlr[r]), o[r]);
    }
  }
  // groups 1.. hand their sums to group 0, which adds them in group order
  if constexpr (WAYS > 1) {
    if (j > 0) *reinterpret_cast<float4*>(&part[j - 1][d]) = acc;  // NOLINT
    __syncthreads();
    if (j > 0) return;
#pragma unroll
    for (int k = 0; k < WAYS - 1; ++k) {
      const float4 p = *reinterpret_cast<const float4*>(&part[k][d]);
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
  }
  const float inv = 1.0f / fmaxf(wsum, 1e-20f);
  if constexpr (E4M3_OUT) {
    // E4M3(o / out_scale), IEEE division, the cache encoder's rounding
    const float s = a.out_scale;
    const uint32_t w4 = e4m3_encode(__fdiv_rn(acc.x * inv, s)) |
                        (e4m3_encode(__fdiv_rn(acc.y * inv, s)) << 8) |
                        (e4m3_encode(__fdiv_rn(acc.z * inv, s)) << 16) |
                        (e4m3_encode(__fdiv_rn(acc.w * inv, s)) << 24);
    *reinterpret_cast<uint32_t*>(a.out8 + static_cast<int64_t>(b) * a.out_stride + h * D + d) =
        w4;
  } else {
    const uint32_t lo01 = static_cast<uint32_t>(f32_to_bf16(acc.x * inv)) |
                          (static_cast<uint32_t>(f32_to_bf16(acc.y * inv)) << 16);
    const uint32_t lo23 = static_cast<uint32_t>(f32_to_bf16(acc.z * inv)) |
                          (static_cast<uint32_t>(f32_to_bf16(acc.w * inv)) << 16);
    *reinterpret_cast<uint2*>(a.out + static_cast<int64_t>(b) * a.out_stride + h * D + d) =
        make_uint2(lo01, lo23);
  }
  // Only now let the next step's partial grid be placed: a combine CTA that
  // lingered beside it would hold registers that the partial kernel's third
  // CTA of an SM needs (three balanced BF16 CTAs take 61,440 of the 65,536).
  asm volatile("griddepcontrol.launch_dependents;");
}

template <int FMT, int D>
cudaError_t launch_simple(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = (static_cast<size_t>(a.group) * D + a.group * kTile + 3 * kMaxGroup) *
                      sizeof(float);
  auto kern = partial_simple_kernel<FMT, D>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(a.num_kv_heads, a.num_splits, a.num_seqs);
  // a programmatic dependent of the previous work on the stream
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT>
cudaError_t launch_simple_fmt(const DecodeArgs& a, int D, cudaStream_t st) {
  switch (D) {
    case 64: return launch_simple<FMT, 64>(a, st);
    case 128: return launch_simple<FMT, 128>(a, st);
    case 256: return launch_simple<FMT, 256>(a, st);
    case 512: return launch_simple<FMT, 512>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_partial(const DecodeArgs& a, int head_dim, int kv_dtype,
                                  cudaStream_t st) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (kv_dtype) {
    case PD_KV_BF16: return launch_simple_fmt<PD_KV_BF16>(a, head_dim, st);
    case PD_KV_FP8_E4M3: return launch_simple_fmt<PD_KV_FP8_E4M3>(a, head_dim, st);
    default: return launch_simple_fmt<PD_KV_NVFP4>(a, head_dim, st);
  }
}

template <int D, int WAYS>
cudaError_t launch_combine_pdl(const CombineArgs& a, cudaStream_t st) {
  // Programmatic dependent launch: the combine grid may be scheduled while the
  // partial kernel drains; griddepcontrol.wait inside keeps it correct.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_q_heads, a.num_seqs);
  cfg.blockDim = dim3(CombineShape<D, WAYS>::kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.out8 != nullptr) return cudaLaunchKernelEx(&cfg, combine_kernel<D, WAYS, true>, a);
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, WAYS, false>, a);
}

// Lane groups for rows of up to max_parts partials: enough that each
// thread's first kRows loads cover them (a power of two), at most 256
// threads a CTA.
template <int D>
cudaError_t launch_combine_ways(const CombineArgs& a, int max_parts, cudaStream_t st) {
  constexpr int kRows = CombineShape<D, 1>::kRows;
  constexpr int kMaxWays = (1024 / D) < 8 ? (1024 / D) : 8;
  int ways = 1;
  while (ways < kMaxWays && ways * kRows < max_parts) ways *= 2;
  if constexpr (kMaxWays >= 8) {
    if (ways == 8) return launch_combine_pdl<D, 8>(a, st);
  }
  if constexpr (kMaxWays >= 4) {
    if (ways == 4) return launch_combine_pdl<D, 4>(a, st);
  }
  if (ways == 2) return launch_combine_pdl<D, 2>(a, st);
  return launch_combine_pdl<D, 1>(a, st);
}

cudaError_t launch_decode_combine(const CombineArgs& a, int head_dim, int max_parts,
                                  cudaStream_t st) {
  if (a.num_seqs == 0) return cudaSuccess;
  cudaError_t e;
  switch (head_dim) {
    case 64: e = launch_combine_ways<64>(a, max_parts, st); break;
    case 128: e = launch_combine_ways<128>(a, max_parts, st); break;
    case 256: e = launch_combine_ways<256>(a, max_parts, st); break;
    case 512: e = launch_combine_ways<512>(a, max_parts, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pd
