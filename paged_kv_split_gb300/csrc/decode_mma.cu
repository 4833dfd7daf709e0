// Split-KV partial kernel on tensor cores with a TMA-fed shared-memory ring.
//
// It computes the split-KV partial of metrale "prefill_attn_b.rs"
// (`paged_decode_attn_splitk_{bf16,fp8,nvfp4}`: each block writes its partial
// output and softmax state to the workspace) for one (sequence, kv head,
// split). The design is this library's own, for sm_103a:
//
//  * One CTA per (kv head, split, sequence) packs the whole GQA group (up to
//    16 q heads), so every K/V byte crosses HBM once per kv head.
//  * Warp 4 is the producer. For each tile of kKT keys it looks up the pages
//    in the block table (one int32 per page; AstrAI "single page-table lookup
//    per tile") and copies each (page, kv head) slab into a ring stage with
//    TMA: a 3-D tiled `cp.async.bulk.tensor` with 128-byte swizzle for the
//    BF16 / FP8 caches ([page][row][head][d] is a regular 3-D tensor of rows),
//    and 1-D `cp.async.bulk` copies (data + scales) for the head-major NVFP4
//    page. Completion is tracked by mbarrier transaction counts; consumers
//    hand stages back through a second mbarrier. Every wait is bounded.
//  * Warps 0-3 consume. The contraction is small (G <= 16 query rows), so it
//    runs on mma.sync m16n8k16 with the operands swapped: S^T = K Q^T puts 16
//    keys on M and 8 q heads on N, O^T = V^T P^T puts 16 head-dim rows on M.
//    P^T is rebuilt as a B fragment from the S^T accumulator with movmatrix.
//    BF16 caches feed ldmatrix directly (bf16 MMA). FP8 / NVFP4 codes are
//    converted in registers to f16, which holds every E4M3 value and every
//    E2M1 x E4M3 product exactly (f16 MMA); q is scaled by a power of two per
//    head into f16 range and the factor is folded into the score multiplier.
//  * head_dim <= 128: each consumer warp owns 16 of the stage's 64 keys over
//    the full head_dim, with its own online-softmax state; the four warps are
//    merged once at the end. head_dim 256 / 512: each warp owns a quarter of
//    head_dim for all keys; partial scores are summed across the warps through
//    shared memory once per 16-key tile.
//  * Keys outside the split's range, in pages whose block-table entry is out
//    of the pool, or past the sequence end are masked: score -inf and V
//    zeroed, so whatever bytes sit in those rows never reach the result.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "pd_common.cuh"

// Cfg<> defines every layout constant for every form; NVFP4 ignores some.
#pragma nv_diag_suppress 177

namespace pd {
namespace {

// Shared-memory budget of the stage ring per CTA (bytes; at least 2 stages):
// 64 KB lets three CTAs share an SM for head_dim <= 128; the head_dim-split
// kernels (256 / 512) do better with 96 KB and two CTAs.
#ifndef PD_MMA_RING_BYTES_SMALL_D
#define PD_MMA_RING_BYTES_SMALL_D (64 * 1024)
#endif
#ifndef PD_MMA_RING_BYTES_LARGE_D
#define PD_MMA_RING_BYTES_LARGE_D (96 * 1024)
#endif

constexpr int kConsumerWarps = 4;
constexpr int kMmaThreads = (kConsumerWarps + 1) * 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; false after ~2 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two E4M3 codes (low byte = first element) -> f16x2 (low half = first). Exact.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// Four bytes, each two E2M1 codes (low nibble = first element) -> four f16x2.
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, uint32_t y) {
  __half2 hx, hy;
  memcpy(&hx, &x, 4);
  memcpy(&hy, &y, 4);
  const __half2 hr = __hmul2(hx, hy);
  uint32_t r;
  memcpy(&r, &hr, 4);
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  uint32_t r;
  memcpy(&r, &h, 4);
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  uint32_t r;
  memcpy(&r, &h, 4);
  return r;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// Load n bytes (4, 8 or 16) from shared memory into words w[0..n/4).
template <int N>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t* w) {
  if constexpr (N == 16) {
    const uint4 v = lds128(addr);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (N == 8) {
    const uint2 v = lds64(addr);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = lds32(addr);
  }
}
// 128-byte swizzle of a byte offset inside a 1024-byte aligned region (the
// pattern TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ ((off >> 3) & 0x70u); }
template <bool ON>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  if constexpr (ON) return swz128(off);
  return off;
}
// 2^e as a float, e clamped to normal exponents.
__device__ __forceinline__ float exp2i(int e) {
  e = e < -120 ? -120 : (e > 120 ? 120 : e);
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}
// floor(log2 |m|) for m > 0 normal; 0 otherwise
__device__ __forceinline__ int ilog2f(float m) {
  return m > 0.0f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127 : 0;
}

// ---------------------------------------------------------------------------
template <int FMT, int D, int NT, int BS>
struct Cfg {
  static constexpr bool kF16 = FMT != PD_KV_BF16;          // MMA operand type
  static constexpr int kDSplit = D <= 128 ? 1 : 4;          // warps sharing head_dim
  static constexpr int kDS = D / kDSplit;                   // head_dim slice per warp (64|128)
  static constexpr int kKSteps = kDS / 16;                  // k-steps of S^T, m-tiles of O^T
  // m-tiles of 16 keys each consumer warp takes per stage (head_dim <= 128),
  // so that a stage carries enough bytes per dependent chain of loads,
  // conversions, MMAs and the softmax update
#ifdef PD_MMA_WM_OVERRIDE
  static constexpr int kWM = PD_MMA_WM_OVERRIDE;
#else
  static constexpr int kWM = 1;  // measured best for every form (one 16-key m-tile per warp)
#endif
  static constexpr int kKT = kDSplit == 1 ? 64 * kWM : 16;  // keys per stage
  static constexpr int kMT = kKT / 16;                      // 16-key m-tiles per stage
  static constexpr int kBR = kKT < BS ? kKT : BS;           // rows per copy
  static constexpr int kNCopy = kKT / kBR;                  // copies per stage and cache
  static constexpr int kRowBytes = FMT == PD_KV_BF16 ? 2 * D : (FMT == PD_KV_FP8_E4M3 ? D : D / 2);
  // BF16 / FP8: each key row is kDCH chunks of kCRB bytes, chunk-major in smem
  static constexpr int kCRB = FMT == PD_KV_NVFP4 ? D / 2 : (kRowBytes < 128 ? kRowBytes : 128);
  static constexpr int kDCH = kRowBytes / kCRB;
  static constexpr int kCopyElems = FMT == PD_KV_BF16 ? kCRB / 2 : kCRB;  // box inner extent
  // 128-byte rows are TMA-swizzled (conflict-free fragment loads); narrower
  // rows (FP8 at head_dim 64) are copied unswizzled
  static constexpr bool kSwizzle = kCRB == 128;
  static constexpr int kDataBytes = kKT * kRowBytes;                       // one cache, one stage
  static constexpr int kScaleBytes = FMT == PD_KV_NVFP4 ? kKT * (D / 16) : 0;
  static constexpr int kCacheStageBytes = (kDataBytes + kScaleBytes + 1023) / 1024 * 1024;
  static constexpr int kStageBytes = 2 * kCacheStageBytes;
  static constexpr int kStagesRaw =
      (kDSplit == 1 ? PD_MMA_RING_BYTES_SMALL_D : PD_MMA_RING_BYTES_LARGE_D) / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  // cross-warp score sums (head_dim split): 2 buffers x 4 warps x m-tiles x 32 lanes x 4*NT
  static constexpr int kRedBytes = kDSplit == 4 ? 2 * 4 * kMT * 32 * 4 * NT * 4 : 0;
  static constexpr int kMergeBytes = kDSplit == 1 ? 4 * (kDS * 8 * NT + 2 * 8 * NT) * 4 : 0;
  static_assert(kMergeBytes <= kRingBytes, "the end-of-CTA merge reuses the ring");
  static constexpr int kQMaxBytes = kDSplit == 4 ? 2 * 4 * 8 * 4 : 0;  // [NT][warp][8] floats
  static constexpr int kBarOffset = kRingBytes + kRedBytes + kQMaxBytes;
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + kStages * 4 + 1024;
  // per copy and cache: bytes landed by TMA
  static constexpr uint32_t kCopyBytes =
      kBR * kRowBytes + (FMT == PD_KV_NVFP4 ? kBR * (D / 16) : 0);
};

template <int FMT, int D, int NT, int BS>
__global__ void __launch_bounds__(kMmaThreads)
    partial_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using C = Cfg<FMT, D, NT, BS>;
  constexpr bool F16 = C::kF16;
  // let the dependent combine grid be scheduled as this grid drains (it waits
  // for this grid's completion before reading the workspace)
  asm volatile("griddepcontrol.launch_dependents;");
  // Launched as a programmatic dependent of whatever came before on the
  // stream (the previous step's combine, say): nothing global is read or
  // written before that grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int g = blockIdx.x;  // kv head
  const int s = blockIdx.y;  // split
  const int b = blockIdx.z;  // sequence
  const int G = a.group;
  const int bs = a.block_size;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int r = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair

  // Without a window the split's first page does not depend on the sequence
  // length, so the producer loads its block-table entries (and prefetches the
  // tensor maps) while the length is still in flight.
  const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  int spec_entry = -1;
  if (warp == kConsumerWarps && a.sliding_window == 0) {
    if constexpr (FMT != PD_KV_NVFP4) {
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      }
    }
    const int e = s * a.chunk + lane;
    if (e < a.max_blocks_per_seq) spec_entry = bt[e];
  }

  // ---- the split's key range ----
  int L = a.seq_lens[b];
  {
    const int cap = a.max_blocks_per_seq * bs;
    if (L < 0 || L > cap) {
      if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
      L = L < 0 ? 0 : cap;
    }
  }
  const int lo = window_lo(L, a.sliding_window);
  const int P = num_key_pages(L, a.sliding_window, bs);
  if (s * a.chunk >= P) {  // no key of this sequence falls in this split
    if (a.direct && P == 0 && s == 0) {  // an empty sequence: zero output rows
      uint16_t* o = a.out + (static_cast<int64_t>(b) * a.num_q_heads + g * G) * D;
      for (int e = tid; e < G * D; e += blockDim.x) o[e] = 0;
    }
    return;
  }
  const int n_act = (P + a.chunk - 1) / a.chunk;  // splits of this sequence that hold keys
  const bool direct = a.direct && n_act == 1;      // this split alone: write the output
  const int first_page = lo / bs + s * a.chunk;
  const int last_page = min(lo / bs + P, first_page + a.chunk);  // exclusive
  const int t_base = first_page * bs;                             // tile origin (page aligned)
  const int t_begin = max(lo, t_base);
  const int t_end = min(L, last_page * bs);
  const int ntiles = (t_end - t_base + C::kKT - 1) / C::kKT;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* ring = smem;
  float* red = reinterpret_cast<float*>(smem + C::kRingBytes);
  float* qmax_s = reinterpret_cast<float*>(smem + C::kRingBytes + C::kRedBytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint32_t* bad_copies = reinterpret_cast<uint32_t*>(empty_bar + C::kStages);

  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // =========================== producer warp ===============================
  if (warp == kConsumerWarps) {
    // entries [cached_base, cached_base + 32) of the block-table row, one per lane
    int cached_base = a.sliding_window == 0 ? s * a.chunk : -(1 << 30);
    int my_entry = spec_entry;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % C::kStages;
      if (i >= C::kStages &&
          !mbar_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) - 1) & 1)) {
        if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
        break;  // consumers give up on their own bounded waits
      }
      const int t0 = t_base + i * C::kKT;
      uint32_t bad = 0;
      uint32_t bytes = 0;
      int pages[C::kNCopy];
#pragma unroll
      for (int j = 0; j < C::kNCopy; ++j) {
        const int tt = t0 + j * C::kBR;
        pages[j] = -1;
        if (tt < t_end) {
          const int pidx = tt / bs;
          if (pidx - cached_base >= 32 || pidx < cached_base) {  // warp-uniform refill
            cached_base = pidx;
            const int e = cached_base + lane;
            my_entry = (e < a.max_blocks_per_seq) ? bt[e] : -1;
          }
          const int pg = __shfl_sync(0xFFFFFFFFu, my_entry, pidx - cached_base);
          if (pg >= 0 && pg < a.num_blocks) {
            pages[j] = pg;
            bytes += 2u * C::kCopyBytes;
          } else {
            bad |= 1u << j;
          }
        }
      }
      const uint32_t fb = smem_u32(&full_bar[st]);
      if (lane == 0) {
        if (bad) atomicOr(a.flags, PD_DEV_BAD_PAGE);
        bad_copies[st] = bad;
        mbar_arrive_expect_tx(fb, bytes);
      }
      __syncwarp();
      // one lane per page issues that page's copies, in parallel
      {
        int my_page = -1;
#pragma unroll
        for (int j = 0; j < C::kNCopy; ++j)
          if (lane == j) my_page = pages[j];
        if (lane < C::kNCopy && my_page >= 0) {
          const int j = lane;
          const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
          const uint32_t vst = kst + C::kCacheStageBytes;
          const int row0 = (t0 + j * C::kBR) % bs;
          if constexpr (FMT == PD_KV_NVFP4) {
            const int64_t line = static_cast<int64_t>(g) * bs + row0;
            const uint8_t* kp = a.k_cache + my_page * a.page_bytes;
            const uint8_t* vp = a.v_cache + my_page * a.page_bytes;
            constexpr uint32_t db = C::kBR * (D / 2);
            constexpr uint32_t sb = C::kBR * (D / 16);
            const uint32_t doff = j * db;
            const uint32_t soff = C::kDataBytes + j * sb;
            bulk_load(kst + doff, kp + line * (D / 2), db, fb);
            bulk_load(vst + doff, vp + line * (D / 2), db, fb);
            bulk_load(kst + soff, kp + a.data_bytes + line * (D / 16), sb, fb);
            bulk_load(vst + soff, vp + a.data_bytes + line * (D / 16), sb, fb);
          } else {
            const int z = my_page * bs + row0;
#pragma unroll
            for (int ch = 0; ch < C::kDCH; ++ch) {
              const uint32_t off = ch * (C::kKT * C::kCRB) + j * (C::kBR * C::kCRB);
              tma_load_3d(kst + off, &tm_k, ch * C::kCopyElems, g, z, fb);
              tma_load_3d(vst + off, &tm_v, ch * C::kCopyElems, g, z, fb);
            }
          }
        }
      }
      __syncwarp();
    }
    return;
  }

  // =========================== consumer warps ==============================
  const int d0 = C::kDSplit == 4 ? warp * C::kDS : 0;  // this warp's head_dim slice

  // ---- q fragments (B operand of S^T = K Q^T), kept in registers ----
  // BF16: natural order, k index = d. f16 forms: thread column c owns the
  // slice's d in [c*DS/4, (c+1)*DS/4); k-step ks uses d = c*DS/4 + 4ks + {0..3}.
  uint32_t qf[C::kKSteps][NT][2];
  float qmul[NT][2];  // score multiplier (log2 units) of the two head columns of this thread
  {
    const uint16_t* qb = a.q + static_cast<int64_t>(b) * a.q_stride + g * G * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + r;  // q head row of the B fragment
      if constexpr (!F16) {
        qmul[nt][0] = qmul[nt][1] = a.scale_log2;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          uint32_t w0 = 0, w1 = 0;
          if (n < G) {
            const uint16_t* p = qb + n * D + d0 + ks * 16 + 2 * c;
            w0 = *reinterpret_cast<const uint32_t*>(p);
            w1 = *reinterpret_cast<const uint32_t*>(p + 8);
          }
          qf[ks][nt][0] = w0;
          qf[ks][nt][1] = w1;
        }
      } else {
        // this thread's q values (4 consecutive d per k-step), loaded up front
        uint2 raw[C::kKSteps];
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks)
          raw[ks] = (n < G) ? *reinterpret_cast<const uint2*>(qb + n * D + d0 + c * (C::kDS / 4) +
                                                               4 * ks)
                            : make_uint2(0u, 0u);
        // power-of-two scale putting max |q| of head n in [2^14, 2^15)
        float m = 0.0f;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks)
          m = fmaxf(fmaxf(m, fmaxf(fabsf(bf16_lo(raw[ks].x)), fabsf(bf16_hi(raw[ks].x)))),
                    fmaxf(fabsf(bf16_lo(raw[ks].y)), fabsf(bf16_hi(raw[ks].y))));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        if constexpr (C::kDSplit == 4) {  // the other warps hold the rest of head_dim
          if (c == 0) qmax_s[(nt * 4 + warp) * 8 + r] = m;
          consumers_sync();
          m = fmaxf(fmaxf(qmax_s[(nt * 4 + 0) * 8 + r], qmax_s[(nt * 4 + 1) * 8 + r]),
                    fmaxf(qmax_s[(nt * 4 + 2) * 8 + r], qmax_s[(nt * 4 + 3) * 8 + r]));
        }
        const float qdown = exp2i(14 - ilog2f(m));
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float mj = __shfl_sync(0xFFFFFFFFu, m, (2 * c + j) * 4);
          qmul[nt][j] = a.scale_log2 * (FMT == PD_KV_FP8_E4M3 ? a.k_scale : 1.0f) *
                        exp2i(ilog2f(mj) - 14);
        }
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          qf[ks][nt][0] = pack_f16x2(bf16_lo(raw[ks].x) * qdown, bf16_hi(raw[ks].x) * qdown);
          qf[ks][nt][1] = pack_f16x2(bf16_lo(raw[ks].y) * qdown, bf16_hi(raw[ks].y) * qdown);
        }
      }
    }
  }

  // ---- running state ----
  float acc[C::kKSteps][NT][4];  // O^T: [head_dim m-tile][n-tile][fragment]
#pragma unroll
  for (int i = 0; i < C::kKSteps; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][nt][k] = 0.0f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.0f;
  }

  bool failed = false;
  int red_buf = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::kStages;
    // after one failed wait, stop waiting (bounded total time); results are
    // then discarded, but every named barrier is still reached
    if (!failed && !mbar_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1)) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      failed = true;
    }
    const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
    const uint32_t vst = kst + C::kCacheStageBytes;
    const uint32_t bad = bad_copies[st];
    const int t0 = t_base + i * C::kKT;

      // ---- scores of one 16-key m-tile over this warp's head_dim slice ----
      auto qk = [&](const int key0, float (&sc)[NT][4]) {
        if constexpr (FMT == PD_KV_BF16) {
          const int mi = lane >> 3, ri = lane & 7;
          const int key = key0 + ri + 8 * (mi & 1);
  #pragma unroll
          for (int ks = 0; ks < C::kKSteps; ++ks) {
            const int d = d0 + ks * 16 + 8 * (mi >> 1);
            const uint32_t off = (d / 64) * (C::kKT * 128) + key * 128 + (d % 64) * 2;
            uint32_t af[4];
            ldsm_x4(kst + swz128(off), af);
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<false>(sc[nt], af, qf[ks][nt][0], qf[ks][nt][1]);
          }
        } else if constexpr (FMT == PD_KV_FP8_E4M3) {
          // keys key0+r, key0+r+8: bytes d in [c*DS/4, +DS/4) = kKSteps words
          uint32_t wa[C::kKSteps], wb[C::kKSteps];
          const int dbyte = d0 + c * (C::kDS / 4);
          const uint32_t base = (dbyte / C::kCRB) * (C::kKT * C::kCRB) + (dbyte % C::kCRB);
  #pragma unroll
          for (int q4 = 0; q4 < C::kKSteps / 4; ++q4) {
            const uint32_t offa = base + (key0 + r) * C::kCRB + 16 * q4;
            lds_words<16>(kst + swz<C::kSwizzle>(offa), wa + 4 * q4);
            lds_words<16>(kst + swz<C::kSwizzle>(offa + 8 * C::kCRB), wb + 4 * q4);
          }
  #pragma unroll
          for (int ks = 0; ks < C::kKSteps; ++ks) {
            uint32_t af[4];
            af[0] = e4m3x2_f16x2(wa[ks] & 0xFFFFu);
            af[1] = e4m3x2_f16x2(wb[ks] & 0xFFFFu);
            af[2] = e4m3x2_f16x2(wa[ks] >> 16);
            af[3] = e4m3x2_f16x2(wb[ks] >> 16);
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<true>(sc[nt], af, qf[ks][nt][0], qf[ks][nt][1]);
          }
        } else {  // NVFP4
          constexpr int kB = C::kDS / 8;  // data bytes of this thread's slice per key (8|16)
          const int dn = d0 + c * (C::kDS / 4);
          const uint32_t offa = (key0 + r) * (D / 2) + dn / 2;
          uint32_t wa[kB / 4], wb[kB / 4];
          lds_words<kB>(kst + offa, wa);
          lds_words<kB>(kst + offa + 8 * (D / 2), wb);
          // one E4M3 scale per 16 elements: k-steps 4j..4j+3 use this slice's group j
          uint32_t sa[C::kKSteps / 4], sbv[C::kKSteps / 4];
          const uint32_t soa = C::kDataBytes + (key0 + r) * (D / 16) + dn / 16;
  #pragma unroll
          for (int j = 0; j < C::kKSteps / 4; ++j) {
            const uint32_t xa = lds_u8(kst + soa + j);
            const uint32_t xb = lds_u8(kst + soa + 8 * (D / 16) + j);
            sa[j] = e4m3x2_f16x2(xa | (xa << 8));
            sbv[j] = e4m3x2_f16x2(xb | (xb << 8));
          }
  #pragma unroll
          for (int w = 0; w < kB / 4; ++w) {
            uint32_t xa[4], xb[4];
            e2m1x8_f16x2(wa[w], xa);
            e2m1x8_f16x2(wb[w], xb);
            // byte 2h of word w -> k-step 2w+h, d +{0,1}; byte 2h+1 -> d +{2,3}
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int ks = 2 * w + h;
              const int grp = ks / 4;
              uint32_t af[4];
              af[0] = hmul2_u32(xa[2 * h], sa[grp]);
              af[1] = hmul2_u32(xb[2 * h], sbv[grp]);
              af[2] = hmul2_u32(xa[2 * h + 1], sa[grp]);
              af[3] = hmul2_u32(xb[2 * h + 1], sbv[grp]);
  #pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma16816<true>(sc[nt], af, qf[ks][nt][0], qf[ks][nt][1]);
            }
          }
        }

      };
      // ---- O^T += V^T P^T for one m-tile (masked keys' V halves zeroed) ----
      // MASKED: the m-tile is ragged, keep_lo / keep_hi zero the V halves of masked keys
      auto pv = [&](auto masked, const int key0, const uint32_t (&pbf)[NT][2],
                    const uint32_t keep_lo, const uint32_t keep_hi) {
        constexpr bool kMasked = decltype(masked)::value;
        if constexpr (FMT == PD_KV_BF16) {
          const int mi = lane >> 3, ri = lane & 7;
          const int key = key0 + ri + 8 * (mi >> 1);
  #pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            const int d = d0 + md * 16 + 8 * (mi & 1);
            const uint32_t off = (d / 64) * (C::kKT * 128) + key * 128 + (d % 64) * 2;
            uint32_t af[4];
            ldsm_x4_trans(vst + swz128(off), af);
            if constexpr (kMasked) {
              af[0] &= keep_lo;
              af[1] &= keep_lo;
              af[2] &= keep_hi;
              af[3] &= keep_hi;
            }
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<false>(acc[md][nt], af, pbf[nt][0], pbf[nt][1]);
          }
        } else if constexpr (FMT == PD_KV_FP8_E4M3) {
          // V bytes d in [r*DS/8, (r+1)*DS/8) of keys 2c, 2c+1, 2c+8, 2c+9; byte j is
          // head_dim row (m-tile j, row r) for j < DS/16 and (j - DS/16, row r+8) above
          constexpr int kVB = C::kDS / 8;  // 16 or 8
          const int dbyte = d0 + r * kVB;
          const uint32_t base = (dbyte / C::kCRB) * (C::kKT * C::kCRB) + (dbyte % C::kCRB);
          uint32_t v[4][kVB / 4];
  #pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int key = key0 + 2 * c + (k4 & 1) + 8 * (k4 >> 1);
            lds_words<kVB>(vst + swz<C::kSwizzle>(base + key * C::kCRB), v[k4]);
          }
          // interleave the bytes of the key pairs: PRMT gives {a_j, b_j, a_j+1, b_j+1}
          uint32_t pr01[kVB / 2], pr23[kVB / 2];
  #pragma unroll
          for (int w = 0; w < kVB / 4; ++w) {
            pr01[2 * w] = __byte_perm(v[0][w], v[1][w], 0x5140);
            pr01[2 * w + 1] = __byte_perm(v[0][w], v[1][w], 0x7362);
            pr23[2 * w] = __byte_perm(v[2][w], v[3][w], 0x5140);
            pr23[2 * w + 1] = __byte_perm(v[2][w], v[3][w], 0x7362);
          }
          // byte pair j sits in pr[j / 2], half j % 2
  #pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            const int jl = md, jh = md + C::kKSteps;
            uint32_t af[4];
            af[0] = e4m3x2_f16x2(pr01[jl >> 1] >> (16 * (jl & 1)));
            af[1] = e4m3x2_f16x2(pr01[jh >> 1] >> (16 * (jh & 1)));
            af[2] = e4m3x2_f16x2(pr23[jl >> 1] >> (16 * (jl & 1)));
            af[3] = e4m3x2_f16x2(pr23[jh >> 1] >> (16 * (jh & 1)));
            if constexpr (kMasked) {
              af[0] &= keep_lo;
              af[1] &= keep_lo;
              af[2] &= keep_hi;
              af[3] &= keep_hi;
            }
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<true>(acc[md][nt], af, pbf[nt][0], pbf[nt][1]);
          }
        } else {  // NVFP4
          // V nibbles d in [r*DS/8, (r+1)*DS/8) of keys 2c, 2c+1, 2c+8, 2c+9 (one scale
          // group per key); nibble j is head_dim row (j, r) below DS/16, else (j - DS/16, r+8)
          constexpr int kVB = C::kDS / 16;  // data bytes per key (8 or 4)
          const int dn = d0 + r * (C::kDS / 8);
          uint32_t v[4][2];
          uint32_t sv[4];
  #pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int key = key0 + 2 * c + (k4 & 1) + 8 * (k4 >> 1);
            v[k4][1] = 0u;
            lds_words<kVB>(vst + key * (D / 2) + dn / 2, v[k4]);
            sv[k4] = lds_u8(vst + C::kDataBytes + key * (D / 16) + dn / 16);
          }
          const uint32_t s01 = e4m3x2_f16x2(sv[0] | (sv[1] << 8));
          const uint32_t s23 = e4m3x2_f16x2(sv[2] | (sv[3] << 8));
          // pair bytes (a_j | b_j << 4): even j from the low nibbles, odd j from the high
          uint32_t f01[2 * kVB], f23[2 * kVB];  // f16x2 per nibble index j
  #pragma unroll
          for (int w = 0; w < kVB / 4; ++w) {
            const uint32_t e01 = (v[0][w] & 0x0F0F0F0Fu) | ((v[1][w] & 0x0F0F0F0Fu) << 4);
            const uint32_t o01 = ((v[0][w] >> 4) & 0x0F0F0F0Fu) | (v[1][w] & 0xF0F0F0F0u);
            const uint32_t e23 = (v[2][w] & 0x0F0F0F0Fu) | ((v[3][w] & 0x0F0F0F0Fu) << 4);
            const uint32_t o23 = ((v[2][w] >> 4) & 0x0F0F0F0Fu) | (v[3][w] & 0xF0F0F0F0u);
            uint32_t t[4];
            e2m1x8_f16x2(e01, t);
  #pragma unroll
            for (int k = 0; k < 4; ++k) f01[8 * w + 2 * k] = hmul2_u32(t[k], s01);
            e2m1x8_f16x2(o01, t);
  #pragma unroll
            for (int k = 0; k < 4; ++k) f01[8 * w + 2 * k + 1] = hmul2_u32(t[k], s01);
            e2m1x8_f16x2(e23, t);
  #pragma unroll
            for (int k = 0; k < 4; ++k) f23[8 * w + 2 * k] = hmul2_u32(t[k], s23);
            e2m1x8_f16x2(o23, t);
  #pragma unroll
            for (int k = 0; k < 4; ++k) f23[8 * w + 2 * k + 1] = hmul2_u32(t[k], s23);
          }
  #pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            uint32_t af[4];
            af[0] = f01[md];
            af[1] = f01[md + C::kKSteps];
            af[2] = f23[md];
            af[3] = f23[md + C::kKSteps];
            if constexpr (kMasked) {
              af[0] &= keep_lo;
              af[1] &= keep_lo;
              af[2] &= keep_hi;
              af[3] &= keep_hi;
            }
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<true>(acc[md][nt], af, pbf[nt][0], pbf[nt][1]);
          }
        }
      };
      auto key_ok = [&](int kk) {  // kk: key index within the stage
        const int kabs = t0 + kk;
        return kabs >= t_begin && kabs < t_end && !((bad >> (kk / C::kBR)) & 1u);
      };
      // m-tiles this warp handles in this stage: its own kWM (keys split across
      // warps) or all of them (head_dim split across warps)
      constexpr int kU = C::kDSplit == 1 ? C::kWM : C::kMT;
      auto mt_of = [&](int u) { return C::kDSplit == 1 ? warp * C::kWM + u : u; };

      float sc[kU][NT][4];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sc[u][nt][0] = sc[u][nt][1] = sc[u][nt][2] = sc[u][nt][3] = 0.0f;
        qk(mt_of(u) * 16, sc[u]);
      }

      // ---------------- sum the head_dim slices (head_dim 256/512) ----------
      if constexpr (C::kDSplit == 4) {
        float* mine = red + (red_buf * 4 + warp) * (kU * NT * 32 * 4);
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            *reinterpret_cast<float4*>(mine + ((u * NT + nt) * 32 + lane) * 4) =
                make_float4(sc[u][nt][0], sc[u][nt][1], sc[u][nt][2], sc[u][nt][3]);
        consumers_sync();
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float4 v = *reinterpret_cast<const float4*>(
                  red + (red_buf * 4 + w) * (kU * NT * 32 * 4) + ((u * NT + nt) * 32 + lane) * 4);
              t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
            sc[u][nt][0] = t.x; sc[u][nt][1] = t.y; sc[u][nt][2] = t.z; sc[u][nt][3] = t.w;
          }
      }

      // ---------------- mask, scale, one online-softmax update ----------------
      // fragment rows r (c0,c1) and r+8 (c2,c3) of m-tile u are keys 16*mt + r, +8
      // an m-tile is ragged if any of its 16 keys is masked (warp-uniform)
      bool ragged[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int key0 = mt_of(u) * 16;
        ragged[u] = (t0 + key0 < t_begin) || (t0 + key0 + 16 > t_end) ||
                    ((bad >> (key0 / C::kBR)) & 1u);
      }
      float p[kU][NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key0 = mt_of(u) * 16;
          const bool va = !ragged[u] || key_ok(key0 + r);
          const bool vb = !ragged[u] || key_ok(key0 + r + 8);
          p[u][nt][0] = va ? sc[u][nt][0] * qmul[nt][0] : -INFINITY;
          p[u][nt][1] = va ? sc[u][nt][1] * qmul[nt][1] : -INFINITY;
          p[u][nt][2] = vb ? sc[u][nt][2] * qmul[nt][0] : -INFINITY;
          p[u][nt][3] = vb ? sc[u][nt][3] * qmul[nt][1] : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(p[u][nt][0], p[u][nt][2]));
          mx1 = fmaxf(mx1, fmaxf(p[u][nt][1], p[u][nt][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
        }
        const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
        // the running max of no column moved: every factor is exactly 1, skip the rescale
        const bool grew = __any_sync(0xFFFFFFFFu, mn0 > m_run[nt][0] || mn1 > m_run[nt][1]);
        const float al0 = (mn0 == -INFINITY) ? 1.0f : ex2(m_run[nt][0] - mn0);
        const float al1 = (mn1 == -INFINITY) ? 1.0f : ex2(m_run[nt][1] - mn1);
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
        float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          p[u][nt][0] = (mn0 == -INFINITY) ? 0.0f : ex2(p[u][nt][0] - mn0);
          p[u][nt][1] = (mn1 == -INFINITY) ? 0.0f : ex2(p[u][nt][1] - mn1);
          p[u][nt][2] = (mn0 == -INFINITY) ? 0.0f : ex2(p[u][nt][2] - mn0);
          p[u][nt][3] = (mn1 == -INFINITY) ? 0.0f : ex2(p[u][nt][3] - mn1);
          ls0 += p[u][nt][0] + p[u][nt][2];
          ls1 += p[u][nt][1] + p[u][nt][3];
        }
        if (grew) {
          l_run[nt][0] *= al0;
          l_run[nt][1] *= al1;
#pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            acc[md][nt][0] *= al0;
            acc[md][nt][1] *= al1;
            acc[md][nt][2] *= al0;
            acc[md][nt][3] *= al1;
          }
        }
        l_run[nt][0] += ls0;
        l_run[nt][1] += ls1;
      }

      // ---------------- O^T += V^T P^T, m-tile by m-tile ----------------
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int key0 = mt_of(u) * 16;
        // P^T as B fragments: the 8x8 blocks have keys as rows, q heads as columns
        uint32_t pbf[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t top = F16 ? pack_f16x2(p[u][nt][0], p[u][nt][1])
                                   : pack_bf16x2(p[u][nt][0], p[u][nt][1]);
          const uint32_t bot = F16 ? pack_f16x2(p[u][nt][2], p[u][nt][3])
                                   : pack_bf16x2(p[u][nt][2], p[u][nt][3]);
          pbf[nt][0] = movmatrix_trans(top);
          pbf[nt][1] = movmatrix_trans(bot);
        }
        if (ragged[u]) {
          const uint32_t keep_lo = (key_ok(key0 + 2 * c) ? 0x0000FFFFu : 0u) |
                                   (key_ok(key0 + 2 * c + 1) ? 0xFFFF0000u : 0u);
          const uint32_t keep_hi = (key_ok(key0 + 2 * c + 8) ? 0x0000FFFFu : 0u) |
                                   (key_ok(key0 + 2 * c + 9) ? 0xFFFF0000u : 0u);
          pv(std::true_type{}, key0, pbf, keep_lo, keep_hi);
        } else {
          pv(std::false_type{}, key0, pbf, 0u, 0u);
        }
      }

    if constexpr (C::kDSplit == 4) red_buf ^= 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
  }

  // ---- finish: full row sums, then write (O / l, m, l) ----
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1)
        l_run[nt][j] += __shfl_xor_sync(0xFFFFFFFFu, l_run[nt][j], o);

  const float vmul = FMT == PD_KV_FP8_E4M3 ? a.v_scale : 1.0f;
  // head_dim index of accumulator element (m-tile md, row half hh: 0 -> r, 1 -> r+8)
  auto drow = [&](int md, int hh) -> int {
    if constexpr (FMT == PD_KV_BF16) return d0 + md * 16 + r + 8 * hh;
    return d0 + r * (C::kDS / 8) + hh * C::kKSteps + md;
  };
  const int64_t row0 = (static_cast<int64_t>(b) * a.num_q_heads + g * G) * a.num_splits + s;

  const int64_t orow0 = (static_cast<int64_t>(b) * a.num_q_heads + g * G) * D;  // out row of head 0
  if constexpr (C::kDSplit == 4) {
    // every warp holds the same (m, l) and its own head_dim slice of O
    if (!failed) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = nt * 8 + 2 * c + j;
          if (h >= G) continue;
          const float inv = vmul / fmaxf(l_run[nt][j], 1e-20f);
          if (direct) {
            uint16_t* o = a.out + orow0 + static_cast<int64_t>(h) * D;
#pragma unroll
            for (int md = 0; md < C::kKSteps; ++md) {
              o[drow(md, 0)] = f32_to_bf16(acc[md][nt][j] * inv);
              o[drow(md, 1)] = f32_to_bf16(acc[md][nt][2 + j] * inv);
            }
            continue;
          }
          float* o = a.ws_o + (row0 + static_cast<int64_t>(h) * a.num_splits) * D;
#pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            o[drow(md, 0)] = acc[md][nt][j] * inv;
            o[drow(md, 1)] = acc[md][nt][2 + j] * inv;
          }
          if (warp == 0 && r == 0)
            a.ws_ml[row0 + static_cast<int64_t>(h) * a.num_splits] =
                make_float2(m_run[nt][j], l_run[nt][j]);
        }
    }
  } else {
    // head_dim <= 128: merge the four warps' (m, l, O) through shared memory
    consumers_sync();  // every warp is done with the ring
    constexpr int kHW = 8 * NT;  // head columns per warp record
    float* mrec = reinterpret_cast<float*>(ring);  // [4][kHW]
    float* lrec = mrec + 4 * kHW;                  // [4][kHW]
    float* orec = lrec + 4 * kHW;                  // [4][D][kHW], unnormalised
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hc = nt * 8 + 2 * c + j;
        if (r == 0) {
          mrec[warp * kHW + hc] = m_run[nt][j];
          lrec[warp * kHW + hc] = l_run[nt][j];
        }
#pragma unroll
        for (int md = 0; md < C::kKSteps; ++md) {
          orec[(warp * D + drow(md, 0)) * kHW + hc] = acc[md][nt][j];
          orec[(warp * D + drow(md, 1)) * kHW + hc] = acc[md][nt][2 + j];
        }
      }
    consumers_sync();
    if (!failed) {
      for (int e = tid; e < G * D; e += kConsumerWarps * 32) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mrec[w * kHW + h]);
        float lsum = 0.0f, o = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float mw = mrec[w * kHW + h];
          const float f = (mw == -INFINITY) ? 0.0f : ex2(mw - M);
          lsum += lrec[w * kHW + h] * f;
          o += orec[(w * D + d) * kHW + h] * f;
        }
        if (direct) {
          a.out[orow0 + e] = f32_to_bf16(o * vmul / fmaxf(lsum, 1e-20f));
          continue;
        }
        a.ws_o[(row0 + static_cast<int64_t>(h) * a.num_splits) * D + d] =
            o * vmul / fmaxf(lsum, 1e-20f);
        if (d == 0) a.ws_ml[row0 + static_cast<int64_t>(h) * a.num_splits] = make_float2(M, lsum);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a BF16 / FP8 cache: dims (d, kv head, pool row), box
// (copy_elems, 1, rows), 128-byte swizzle for 128-byte rows.
bool encode_cache_map(CUtensorMap* m, const void* base, int kv_dtype, int D, int hkv,
                      int64_t pool_rows, int copy_elems, int rows, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int esz = kv_dtype == PD_KV_BF16 ? 2 : 1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(hkv),
                              static_cast<cuuint64_t>(pool_rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz,
                                 static_cast<cuuint64_t>(hkv) * D * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(copy_elems), 1u,
                             static_cast<cuuint32_t>(rows)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult rc = fn(
      m, esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
      // L2 fills no wider than one head's row: a wider fill would pull in the
      // next head's bytes, which another CTA reads at some other time
      D * esz >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                     : (D * esz >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                       : CU_TENSOR_MAP_L2_PROMOTION_L2_64B),
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

template <int FMT, int D, int NT, int BS>
cudaError_t launch_mma_cfg(const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<FMT, D, NT, BS>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if constexpr (FMT != PD_KV_NVFP4) {
    const int64_t rows = a.num_blocks * a.block_size;
    if (!encode_cache_map(&tk, a.k_cache, FMT, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          C::kSwizzle) ||
        !encode_cache_map(&tv, a.v_cache, FMT, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          C::kSwizzle))
      return cudaErrorInvalidValue;
  }
  auto kern = partial_mma_kernel<FMT, D, NT, BS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const dim3 grid(a.num_kv_heads, a.num_splits, a.num_seqs);
  // a programmatic dependent of the previous work on the stream
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

template <int FMT, int D, int NT>
cudaError_t launch_mma_bs(const DecodeArgs& a, cudaStream_t st) {
  return a.block_size == 16 ? launch_mma_cfg<FMT, D, NT, 16>(a, st)
                            : launch_mma_cfg<FMT, D, NT, 32>(a, st);
}

template <int FMT, int D>
cudaError_t launch_mma_nt(const DecodeArgs& a, cudaStream_t st) {
  return a.group <= 8 ? launch_mma_bs<FMT, D, 1>(a, st) : launch_mma_bs<FMT, D, 2>(a, st);
}

template <int FMT>
cudaError_t launch_mma_fmt(const DecodeArgs& a, int D, cudaStream_t st) {
  switch (D) {
    case 64: return launch_mma_nt<FMT, 64>(a, st);
    case 128: return launch_mma_nt<FMT, 128>(a, st);
    case 256: return launch_mma_nt<FMT, 256>(a, st);
    case 512: return launch_mma_nt<FMT, 512>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int mma_ctas_per_sm_estimate(int kv_dtype, int head_dim) {
  auto per_sm = [](int smem) { return (227 * 1024) / (smem + 1024); };
  int smem;
  if (kv_dtype == PD_KV_BF16) {
    smem = head_dim <= 128 ? Cfg<PD_KV_BF16, 128, 1, 16>::kSmemBytes
                           : Cfg<PD_KV_BF16, 512, 1, 16>::kSmemBytes;
  } else if (kv_dtype == PD_KV_FP8_E4M3) {
    smem = head_dim <= 128 ? Cfg<PD_KV_FP8_E4M3, 128, 1, 16>::kSmemBytes
                           : Cfg<PD_KV_FP8_E4M3, 512, 1, 16>::kSmemBytes;
  } else {
    smem = head_dim <= 128 ? Cfg<PD_KV_NVFP4, 128, 1, 16>::kSmemBytes
                           : Cfg<PD_KV_NVFP4, 512, 1, 16>::kSmemBytes;
  }
  const int n = per_sm(smem);
  return n < 1 ? 1 : (n > 4 ? 4 : n);
}

cudaError_t launch_decode_partial_mma(const DecodeArgs& a, int head_dim, int kv_dtype,
                                      cudaStream_t st) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (kv_dtype) {
    case PD_KV_BF16: return launch_mma_fmt<PD_KV_BF16>(a, head_dim, st);
    case PD_KV_FP8_E4M3: return launch_mma_fmt<PD_KV_FP8_E4M3>(a, head_dim, st);
    default: return launch_mma_fmt<PD_KV_NVFP4>(a, head_dim, st);
  }
}

}  // namespace pd
