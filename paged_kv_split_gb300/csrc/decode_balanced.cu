// Balanced split-KV partial kernel: the same tensor-core tile pipeline as
// decode_mma.cu, but each CTA walks a host-made plan of "pieces" instead of one
// (sequence, kv head, split).
//
// The host cuts the line of all (sequence, kv head) key-page ranges, laid end
// to end, into one equal share per resident CTA, so every CTA streams the same
// number of pages and the grid is a single generation; a share that crosses a
// (sequence, kv head) boundary becomes several pieces, each with its own
// partial (O, m, l) in the workspace, merged by the combine like split-KV
// partials (metrale "prefill_attn_b.rs" `paged_decode_attn_splitk_*` /
// `paged_decode_attn_reduce_*`: partial output and softmax state per split,
// then a log-sum-exp reduce). A (sequence, kv head) that one piece covers is
// written to the bf16 output directly.
//
//  * Warp 4 produces: for each piece it reads the descriptor (fetched 32 at a
//    time), the piece's block-table entries, copies the GQA group's q rows into
//    a q slot with the piece's first tile, then the K/V pages tile by tile
//    through the stage ring (TMA tensor copies for BF16 / FP8, bulk copies for
//    NVFP4), each stage carrying a record of its piece and key range.
//  * Warps 0-3 consume as in decode_mma.cu (mma.sync with keys on M, q heads
//    on N, online softmax in log2 units). At the end of a piece the four
//    warps merge their (m, l, O) in the stage of the piece's last tile, which
//    they hand back afterwards, and write the piece's partial or output row.
//  * Every consumer barrier is an mbarrier with a bounded wait, and every
//    wait gives up after ~2 s with a device status bit, so a stalled CTA
//    ends with an error instead of hanging.
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
// The same wait taken by a whole warp with one outcome for all its lanes
// (false if any lane ran out of time or `abort_flag` is set), so that the
// warp never splits on a wait that ends near its limit.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort_flag) {
  (void)abort_flag;
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity));
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
// Per-stage record the producer writes before arming the stage's full barrier
// (the consumers read it after their wait on that barrier).
struct StageMeta {
  int b, g, s;          // sequence, kv head and split of the item the tile belongs to
  int t0;               // key index of the tile's first row
  int t_begin, t_end;   // the item's key range [t_begin, t_end)
  uint32_t bad;         // bit j: copy j's page was outside the pool (its keys are masked)
  uint32_t flags;       // kMeta* bits; bits 8.. the item's q slot
};
constexpr uint32_t kMetaFirst = 1u;   // first tile of an item (q landed with it)
constexpr uint32_t kMetaLast = 2u;    // last tile of an item
constexpr uint32_t kMetaDirect = 4u;  // the item is its sequence's only split: write out
constexpr uint32_t kMetaEnd = 8u;     // no more items: consumers leave

template <int FMT, int D, int NT, int BS>
struct Cfg {
  static constexpr bool kF16 = FMT != PD_KV_BF16;          // MMA operand type
  static constexpr int kDSplit = D <= 128 ? 1 : 4;          // warps sharing head_dim
  static constexpr int kDS = D / kDSplit;                   // head_dim slice per warp (64|128)
  static constexpr int kKSteps = kDS / 16;                  // k-steps of S^T, m-tiles of O^T
  // m-tiles of 16 keys each consumer warp takes per stage (head_dim <= 128)
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
  static constexpr int kQMaxBytes = kDSplit == 4 ? NT * 4 * 8 * 4 : 0;  // [NT][warp][8] floats
  static constexpr int kHW = 8 * NT;                        // q-head columns of the tiles
  static constexpr int kMStride = D + 4;                    // floats per merge-slice row
  // end-of-item merge (head_dim <= 128): a [kHW][D+4] slice, per-warp m and l
  // (two buffers, by item parity), and the merged m and l of each column
  static constexpr int kMergeBytes =
      kDSplit == 1 ? (kHW * kMStride + 2 * 2 * 4 * kHW + 2 * kHW) * 4 : 0;
  static constexpr int kQSlots = kDSplit == 1 ? 2 : 1;      // q of the next item lands early
  static constexpr int kMergeOffset = kRingBytes + kRedBytes + kQMaxBytes;
  static constexpr int kMetaOffset = (kMergeOffset + kMergeBytes + 15) / 16 * 16;
  static constexpr int kBarOffset = kMetaOffset + kStages * static_cast<int>(sizeof(StageMeta));
  // full[kStages], empty[kStages], qempty[kQSlots], one consumer barrier
  static constexpr int kNumBars = 2 * kStages + kQSlots + 1;
  static constexpr int kAbortOffset = kBarOffset + kNumBars * 8;
  static constexpr int kQOffset = (kAbortOffset + 16 + 127) / 128 * 128;
  // per copy and cache: bytes landed by TMA
  static constexpr uint32_t kCopyBytes =
      kBR * kRowBytes + (FMT == PD_KV_NVFP4 ? kBR * (D / 16) : 0);
  // dynamic shared memory for a GQA group of G heads (q slots of G rows),
  // with 1 KB of slack for aligning the ring to 1024 bytes
  static constexpr int smem_bytes(int G) { return kQOffset + kQSlots * G * D * 2 + 1024; }
};

// Consumer-warp barrier on an mbarrier (one arrival per warp, bounded wait),
// so that a stalled peer ends in an error instead of a hang.
// Named barrier 1 over the four consumer warps that also ANDs a predicate
// across them: every consumer thread gets the same answer.
__device__ __forceinline__ bool consumers_vote(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
struct ConsumerSync {
  uint32_t bar;
  uint32_t parity;
  volatile int* abort_flag;
  // false if the wait ran out or another warp gave up; the caller then stops
  __device__ __forceinline__ bool operator()(int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, parity, abort_flag);
    parity ^= 1u;
    if (!ok) *abort_flag = 1;
    return ok;
  }
};

template <int FMT, int D, int NT, int BS>
__global__ void __launch_bounds__(kMmaThreads)
    partial_balanced_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using C = Cfg<FMT, D, NT, BS>;
  constexpr bool F16 = C::kF16;
  // let the dependent combine grid be scheduled as this grid drains (it waits
  // for this grid's completion before reading the workspace)
  asm volatile("griddepcontrol.launch_dependents;");
  const int G = a.group;
  const int bs = a.block_size;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int r = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair
  const uint32_t q_bytes = static_cast<uint32_t>(G) * D * 2;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* ring = smem;
  float* red = reinterpret_cast<float*>(smem + C::kRingBytes);
  float* qmax_s = reinterpret_cast<float*>(smem + C::kRingBytes + C::kRedBytes);
  float* mslice = reinterpret_cast<float*>(smem + C::kMergeOffset);  // [kHW][D+4]
  float* mrec = mslice + C::kHW * C::kMStride;                        // [2][4][kHW]
  float* lrec = mrec + 2 * 4 * C::kHW;                                // [2][4][kHW]
  float* fin_m = lrec + 2 * 4 * C::kHW;                               // [kHW]
  float* fin_l = fin_m + C::kHW;                                      // [kHW]
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + C::kMetaOffset);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* qempty_bar = empty_bar + C::kStages;
  uint64_t* cons_bar = qempty_bar + C::kQSlots;
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::kAbortOffset);
  unsigned char* qslots = smem + C::kQOffset;

  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kConsumerWarps);
    }
    for (int i = 0; i < C::kQSlots; ++i) mbar_init(smem_u32(&qempty_bar[i]), kConsumerWarps);
    mbar_init(smem_u32(cons_bar), kConsumerWarps);
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // =========================== producer warp ===============================
  if (warp == kConsumerWarps) {
    if constexpr (FMT != PD_KV_NVFP4) {
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      }
    }
    // this CTA's pieces [p_begin, p_end); lane l holds descriptor desc_base + l
    int p_begin = a.plan_cta[blockIdx.x];
    int p_end = a.plan_cta[blockIdx.x + 1];
    if (p_begin < 0 || p_end > a.plan_num_pieces || p_end < p_begin) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_BAD_PLAN);
      p_begin = p_end = 0;
    }
    int desc_base = p_begin;
    int4 my_desc = make_int4(0, 0, 0, 0);
    if (p_begin + lane < p_end) my_desc = a.plan_pieces[p_begin + lane];
    int i = 0;      // tiles issued
    int k = 0;      // pieces started (q slot k % kQSlots)
    bool ok = true;
    for (int piece = p_begin; piece < p_end && ok; ++piece) {
      if (piece - desc_base >= 32) {  // warp-uniform refill of the descriptor window
        desc_base = piece;
        my_desc = piece + lane < p_end ? a.plan_pieces[piece + lane] : make_int4(0, 0, 0, 0);
      }
      const int src = piece - desc_base;
      const int seg = __shfl_sync(0xFFFFFFFFu, my_desc.x, src);
      const int t_begin = __shfl_sync(0xFFFFFFFFu, my_desc.y, src);
      const int t_end = __shfl_sync(0xFFFFFFFFu, my_desc.z, src);
      const int pflags = __shfl_sync(0xFFFFFFFFu, my_desc.w, src);
      if (seg < 0 || seg >= a.num_seqs * a.num_kv_heads || t_begin < 0 || t_end <= t_begin ||
          t_end > a.max_blocks_per_seq * bs) {  // not a piece this plan can hold: skipped
        if (lane == 0) atomicOr(a.flags, PD_DEV_BAD_PLAN);
        continue;
      }
      const int b = seg / a.num_kv_heads;
      const int g = seg - b * a.num_kv_heads;
      const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
      const int first_page = t_begin / bs;
      int cached_base = first_page;
      int my_entry = (first_page + lane < a.max_blocks_per_seq) ? bt[first_page + lane] : -1;
      {
        const int s = piece;  // the piece's slot in the workspace
        const int t_base = first_page * bs;  // page aligned
        const int ntiles = (t_end - t_base + C::kKT - 1) / C::kKT;
        const int qslot = k % C::kQSlots;
        // the q slot is free once the consumers have read the piece that used it last
        if (k >= C::kQSlots &&
            !warp_wait(smem_u32(&qempty_bar[qslot]), ((k / C::kQSlots) - 1) & 1, abort_s)) {
          ok = false;
          break;
        }
        const uint32_t item_flags = ((pflags & 1) ? kMetaDirect : 0u) |
                                    (static_cast<uint32_t>(qslot) << 8);
        for (int j = 0; j < ntiles; ++j, ++i) {
          const int st = i % C::kStages;
          if (i >= C::kStages &&
              !warp_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) - 1) & 1, abort_s)) {
            ok = false;
            break;
          }
          const int t0 = t_base + j * C::kKT;
          uint32_t bad = 0;
          uint32_t bytes = 0;
          int pages[C::kNCopy];
#pragma unroll
          for (int jj = 0; jj < C::kNCopy; ++jj) {
            const int tt = t0 + jj * C::kBR;
            pages[jj] = -1;
            if (tt < t_end) {
              const int pidx = tt / bs;
              if (pidx - cached_base >= 32 || pidx < cached_base) {  // warp-uniform refill
                cached_base = pidx;
                const int e = cached_base + lane;
                my_entry = (e < a.max_blocks_per_seq) ? bt[e] : -1;
              }
              const int pg = __shfl_sync(0xFFFFFFFFu, my_entry, pidx - cached_base);
              if (pg >= 0 && pg < a.num_blocks) {
                pages[jj] = pg;
                bytes += 2u * C::kCopyBytes;
              } else {
                bad |= 1u << jj;
              }
            }
          }
          if (j == 0) bytes += q_bytes;
          const uint32_t fb = smem_u32(&full_bar[st]);
          if (lane == 0) {
            if (bad) atomicOr(a.flags, PD_DEV_BAD_PAGE);
            StageMeta& m = meta[st];
            m.b = b;
            m.g = g;
            m.s = s;
            m.t0 = t0;
            m.t_begin = t_begin;
            m.t_end = t_end;
            m.bad = bad;
            m.flags = item_flags | (j == 0 ? kMetaFirst : 0u) | (j == ntiles - 1 ? kMetaLast : 0u);
            mbar_arrive_expect_tx(fb, bytes);
          }
          __syncwarp();
          // q rows of the item ride with its first tile (one lane); one lane
          // per page issues that page's copies, in parallel
          if (j == 0 && lane == 31) {
            const uint16_t* qsrc = a.q + static_cast<int64_t>(b) * a.q_stride + g * G * D;
            bulk_load(smem_u32(qslots + qslot * q_bytes), qsrc, q_bytes, fb);
          }
          {
            int my_page = -1;
#pragma unroll
            for (int jj = 0; jj < C::kNCopy; ++jj)
              if (lane == jj) my_page = pages[jj];
            if (lane < C::kNCopy && my_page >= 0) {
              const int jj = lane;
              const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
              const uint32_t vst = kst + C::kCacheStageBytes;
              const int row0 = (t0 + jj * C::kBR) % bs;
              if constexpr (FMT == PD_KV_NVFP4) {
                const int64_t line = static_cast<int64_t>(g) * bs + row0;
                const uint8_t* kp = a.k_cache + my_page * a.page_bytes;
                const uint8_t* vp = a.v_cache + my_page * a.page_bytes;
                constexpr uint32_t db = C::kBR * (D / 2);
                constexpr uint32_t sb = C::kBR * (D / 16);
                const uint32_t doff = jj * db;
                const uint32_t soff = C::kDataBytes + jj * sb;
                bulk_load(kst + doff, kp + line * (D / 2), db, fb);
                bulk_load(vst + doff, vp + line * (D / 2), db, fb);
                bulk_load(kst + soff, kp + a.data_bytes + line * (D / 16), sb, fb);
                bulk_load(vst + soff, vp + a.data_bytes + line * (D / 16), sb, fb);
              } else {
                const int z = my_page * bs + row0;
#pragma unroll
                for (int ch = 0; ch < C::kDCH; ++ch) {
                  const uint32_t off = ch * (C::kKT * C::kCRB) + jj * (C::kBR * C::kCRB);
                  tma_load_3d(kst + off, &tm_k, ch * C::kCopyElems, g, z, fb);
                  tma_load_3d(vst + off, &tm_v, ch * C::kCopyElems, g, z, fb);
                }
              }
            }
          }
          __syncwarp();
        }
        ++k;
      }
    }
    if (ok) {
      // end marker: a stage with no copies whose record tells the consumers to leave
      const int st = i % C::kStages;
      if (i >= C::kStages &&
          !warp_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) - 1) & 1, abort_s)) {
        ok = false;
      } else {
        if (lane == 0) {
          meta[st].flags = kMetaEnd;
          mbar_arrive(smem_u32(&full_bar[st]));
        }
        ++i;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      *abort_s = 1;
      // let the copies already issued land before the block can exit
      for (int t = max(0, i - C::kStages); t < i; ++t)
        (void)mbar_wait(smem_u32(&full_bar[t % C::kStages]), (t / C::kStages) & 1);
    }
    return;
  }

  // =========================== consumer warps ==============================
  const int d0 = C::kDSplit == 4 ? warp * C::kDS : 0;  // this warp's head_dim slice
  ConsumerSync csync{smem_u32(cons_bar), 0u, abort_s};
  const float vmul = FMT == PD_KV_FP8_E4M3 ? a.v_scale : 1.0f;
  // head_dim index of accumulator element (m-tile md, row half hh: 0 -> r, 1 -> r+8)
  auto drow = [&](int md, int hh) -> int {
    if constexpr (FMT == PD_KV_BF16) return d0 + md * 16 + r + 8 * hh;
    return d0 + r * (C::kDS / 8) + hh * C::kKSteps + md;
  };

  int i = 0;  // tiles consumed
  int red_buf = 0;
  int ip = 0;  // item parity (merge buffers)
  bool aborted = false;
  while (!aborted) {
    int st = i % C::kStages;
    {
      bool ok = warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s);
      // head_dim split: the warps meet at named barriers every tile, so they
      // must agree on every wait's outcome before reading the stage record
      if constexpr (C::kDSplit == 4) ok = consumers_vote(ok);
      if (!ok) {
        aborted = true;
        break;
      }
    }
    uint32_t flags = meta[st].flags;
    if (flags & kMetaEnd) break;
    const int b = meta[st].b;
    const int g = meta[st].g;
    const int s = meta[st].s;
    const int t_begin = meta[st].t_begin;
    const int t_end = meta[st].t_end;
    const bool direct = (flags & kMetaDirect) != 0;
    const int qslot = static_cast<int>(flags >> 8);

    // ---- q fragments (B operand of S^T = K Q^T) from the item's q slot ----
    // BF16: natural order, k index = d. f16 forms: thread column c owns the
    // slice's d in [c*DS/4, (c+1)*DS/4); k-step ks uses d = c*DS/4 + 4ks + {0..3}.
    uint32_t qf[C::kKSteps][NT][2];
    float qmul[NT][2];  // score multiplier (log2 units) of the two head columns of this thread
    {
      const uint16_t* qb = reinterpret_cast<const uint16_t*>(qslots + qslot * q_bytes);
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
          // this thread's q values (4 consecutive d per k-step)
          uint2 raw[C::kKSteps];
#pragma unroll
          for (int ks = 0; ks < C::kKSteps; ++ks)
            raw[ks] = (n < G) ? *reinterpret_cast<const uint2*>(qb + n * D + d0 +
                                                                 c * (C::kDS / 4) + 4 * ks)
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
            consumers_bar();  // uniform: the warps agreed on this tile's wait
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
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&qempty_bar[qslot]));

    // ---- running state of the item ----
    float acc[C::kKSteps][NT][4];  // O^T: [head_dim m-tile][n-tile][fragment]
#pragma unroll
    for (int ii = 0; ii < C::kKSteps; ++ii)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) acc[ii][nt][kk] = 0.0f;
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.0f;
    }

    // ---- the item's tiles ----
    while (true) {
    const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
    const uint32_t vst = kst + C::kCacheStageBytes;
    const uint32_t bad = meta[st].bad;
    const int t0 = meta[st].t0;
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
        consumers_bar();  // uniform: the warps agreed on this tile's wait
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
    const bool last = (flags & kMetaLast) != 0;
    // head_dim <= 128: the item's last stage is handed back after the merge,
    // which may use its memory
    const bool hold = C::kDSplit == 1 && last;
    __syncwarp();
    if (lane == 0 && !hold) mbar_arrive(smem_u32(&empty_bar[st]));
    ++i;
    if (last || aborted) break;
    st = i % C::kStages;
    {
      bool ok = warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s);
      if constexpr (C::kDSplit == 4) ok = consumers_vote(ok);
      if (!ok) {
        aborted = true;
        break;
      }
    }
    flags = meta[st].flags;
    }  // tiles of the item
    if (aborted) break;

    // ---- end of the item: full row sums, then write (O / l, m, l) ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1)
          l_run[nt][j] += __shfl_xor_sync(0xFFFFFFFFu, l_run[nt][j], o);

    const int64_t prow = static_cast<int64_t>(s) * G;  // the piece's first (m, l) slot
    const int64_t orow0 = (static_cast<int64_t>(b) * a.num_q_heads + g * G) * D;  // head 0's row
    if constexpr (C::kDSplit == 4) {
      // every warp holds the same (m, l) and its own head_dim slice of O
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
          float* o = a.ws_o + (prow + h) * D;
#pragma unroll
          for (int md = 0; md < C::kKSteps; ++md) {
            o[drow(md, 0)] = acc[md][nt][j] * inv;
            o[drow(md, 1)] = acc[md][nt][2 + j] * inv;
          }
          if (warp == 0 && r == 0)
            a.ws_ml[prow + h] =
                make_float2(m_run[nt][j], l_run[nt][j]);
        }
    } else {
      // head_dim <= 128: merge the four warps' (m, l, O). Per-warp m and l go
      // to a buffer picked by item parity (a warp can reach the next item's
      // merge while another still reads this one's).
      float* mr = mrec + ip * 4 * C::kHW;
      float* lr = lrec + ip * 4 * C::kHW;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hc = nt * 8 + 2 * c + j;
          if (r == 0) {
            mr[warp * C::kHW + hc] = m_run[nt][j];
            lr[warp * C::kHW + hc] = l_run[nt][j];
          }
        }
      const int ostride = D + 4;  // padded rows: conflict-free fragment stores
      if (4 * G * ostride * 4 <= C::kStageBytes) {
        // the four warps' unscaled O in the held stage [warp][head][D+4] (once
        // every warp is done reading its keys), then every thread merges whole
        // output elements (warps 0..3 in order)
        float* orec = reinterpret_cast<float*>(ring + st * C::kStageBytes);
        if (!csync(lane)) break;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int hc = nt * 8 + 2 * c + j;
            if (hc >= G) continue;  // padding columns of the tile
            float* row = orec + (warp * G + hc) * ostride;
#pragma unroll
            for (int md = 0; md < C::kKSteps; ++md)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) row[drow(md, hh)] = acc[md][nt][2 * hh + j];
          }
        if (!csync(lane)) break;
        for (int e = tid; e < G * D; e += kConsumerWarps * 32) {
          const int h = e / D, d = e % D;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) M = fmaxf(M, mr[w * C::kHW + h]);
          float lsum = 0.0f, o = 0.0f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float mw = mr[w * C::kHW + h];
            const float f = (mw == -INFINITY) ? 0.0f : ex2(mw - M);
            lsum += lr[w * C::kHW + h] * f;
            o += orec[(w * G + h) * ostride + d] * f;
          }
          const float v = o * vmul / fmaxf(lsum, 1e-20f);
          if (direct) {
            a.out[orow0 + e] = f32_to_bf16(v);
            continue;
          }
          a.ws_o[(prow + h) * D + d] = v;
          if (d == 0) a.ws_ml[prow + h] = make_float2(M, lsum);
        }
      } else {
        // too large for one stage: accumulate through the merge slice in a
        // fixed order (warp 3, 2, 1, then 0)
        if (!csync(lane)) break;
        float fw[NT][2];  // this warp's factor per column
        float mcol[NT][2], lcol[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int hc = nt * 8 + 2 * c + j;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) M = fmaxf(M, mr[w * C::kHW + hc]);
            float lsum = 0.0f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float mw = mr[w * C::kHW + hc];
              lsum += lr[w * C::kHW + hc] * ((mw == -INFINITY) ? 0.0f : ex2(mw - M));
            }
            fw[nt][j] = (m_run[nt][j] == -INFINITY) ? 0.0f : ex2(m_run[nt][j] - M);
            mcol[nt][j] = M;
            lcol[nt][j] = lsum;
          }
        bool ok = true;
#pragma unroll
        for (int w = 3; w >= 0; --w) {
          if (warp == w) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int hc = nt * 8 + 2 * c + j;
                if (hc >= G) continue;  // padding columns of the tile
                float* row = mslice + hc * C::kMStride;
                const float inv = vmul / fmaxf(lcol[nt][j], 1e-20f);
#pragma unroll
                for (int md = 0; md < C::kKSteps; ++md)
#pragma unroll
                  for (int hh = 0; hh < 2; ++hh) {
                    const int d = drow(md, hh);
                    const float v = acc[md][nt][2 * hh + j] * fw[nt][j];
                    if (w == 3) row[d] = v;
                    else if (w > 0) row[d] += v;
                    else row[d] = (row[d] + v) * inv;  // warp 0 last: normalised
                  }
                if (w == 0 && r == 0) {
                  fin_m[hc] = mcol[nt][j];
                  fin_l[hc] = lcol[nt][j];
                }
              }
          }
          ok = csync(lane) && ok;
        }
        if (!ok) break;
        for (int e = tid; e < G * D; e += kConsumerWarps * 32) {
          const int h = e / D, d = e % D;
          const float v = mslice[h * C::kMStride + d];
          if (direct) {
            a.out[orow0 + e] = f32_to_bf16(v);
            continue;
          }
          a.ws_o[(prow + h) * D + d] = v;
          if (d == 0)
            a.ws_ml[prow + h] =
                make_float2(fin_m[h], fin_l[h]);
        }
      }
      // hand the held stage back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
      ip ^= 1;
    }
  }  // items
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
cudaError_t launch_bal_cfg(const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<FMT, D, NT, BS>;
  const int smem = C::smem_bytes(a.group);
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
  auto kern = partial_balanced_kernel<FMT, D, NT, BS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // per device: the shared-memory limit, set once for the largest group this
  // instantiation serves (concurrent first calls may both set it: harmless)
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::smem_bytes(8 * NT));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // An ordinary launch, not a programmatic dependent: the plan gives every
  // CTA an equal share on the assumption that all of them start together, and
  // a CTA launched early next to the previous step's combine grid may find no
  // room and start a whole share late (measured: 62.6 -> 93 us on the
  // llama8b batch).
  kern<<<a.plan_num_ctas, kMmaThreads, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int FMT, int D, int NT>
cudaError_t launch_bal_bs(const DecodeArgs& a, cudaStream_t st) {
  return a.block_size == 16 ? launch_bal_cfg<FMT, D, NT, 16>(a, st)
                            : launch_bal_cfg<FMT, D, NT, 32>(a, st);
}

template <int FMT, int D>
cudaError_t launch_bal_nt(const DecodeArgs& a, cudaStream_t st) {
  return a.group <= 8 ? launch_bal_bs<FMT, D, 1>(a, st) : launch_bal_bs<FMT, D, 2>(a, st);
}

template <int FMT>
cudaError_t launch_bal_fmt(const DecodeArgs& a, int D, cudaStream_t st) {
  switch (D) {
    case 64: return launch_bal_nt<FMT, 64>(a, st);
    case 128: return launch_bal_nt<FMT, 128>(a, st);
    case 256: return launch_bal_nt<FMT, 256>(a, st);
    case 512: return launch_bal_nt<FMT, 512>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int balanced_ctas_per_sm(int kv_dtype, int head_dim, int group) {
  auto per_sm = [](int smem) { return (228 * 1024) / (smem + 1024); };
  const bool two = group > 8;  // two 8-column n-tiles
  int smem;
#define PD_BAL_SMEM(F, DD) \
  (two ? Cfg<F, DD, 2, 16>::smem_bytes(group) : Cfg<F, DD, 1, 16>::smem_bytes(group))
#define PD_BAL_SMEM_D(F)                                                            \
  (head_dim <= 64 ? PD_BAL_SMEM(F, 64)                                              \
                  : head_dim <= 128 ? PD_BAL_SMEM(F, 128)                           \
                                    : head_dim <= 256 ? PD_BAL_SMEM(F, 256) : PD_BAL_SMEM(F, 512))
  if (kv_dtype == PD_KV_BF16) smem = PD_BAL_SMEM_D(PD_KV_BF16);
  else if (kv_dtype == PD_KV_FP8_E4M3) smem = PD_BAL_SMEM_D(PD_KV_FP8_E4M3);
  else smem = PD_BAL_SMEM_D(PD_KV_NVFP4);
#undef PD_BAL_SMEM_D
#undef PD_BAL_SMEM
  const int n = per_sm(smem);
  return n < 1 ? 1 : (n > 4 ? 4 : n);
}

cudaError_t launch_decode_partial_balanced(const DecodeArgs& a, int head_dim, int kv_dtype,
                                           cudaStream_t st) {
  if (a.num_seqs == 0 || a.plan_num_ctas == 0) return cudaSuccess;
  switch (kv_dtype) {
    case PD_KV_BF16: return launch_bal_fmt<PD_KV_BF16>(a, head_dim, st);
    case PD_KV_FP8_E4M3: return launch_bal_fmt<PD_KV_FP8_E4M3>(a, head_dim, st);
    default: return launch_bal_fmt<PD_KV_NVFP4>(a, head_dim, st);
  }
}

}  // namespace pd
