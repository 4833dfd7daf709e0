// Building blocks shared by the tensor-core partial kernels (decode_mma.cu,
// decode_balanced.cu): PTX wrappers for mbarriers, TMA and bulk copies,
// ldmatrix / mma.sync / movmatrix and the E4M3 / E2M1 conversions, the
// bounded waits, and the host-side tensor-map encoding of a paged cache.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "pd_common.cuh"

namespace pd {
namespace mma {

// Shared-memory budget of the stage ring per CTA (bytes; at least 2 stages):
// 64 KB lets three CTAs share an SM for head_dim <= 128; the head_dim-split
// kernels do better with 96 KB and two CTAs at head_dim 512, and the split
// kernel with 64 KB and three CTAs at 256 (window D=256 workload: 28.3 ->
// 26.9 us; wide D=512 with 64 KB: 48.0 -> 49.1).
#ifndef PD_MMA_RING_BYTES_SMALL_D
#define PD_MMA_RING_BYTES_SMALL_D (64 * 1024)
#endif
#ifndef PD_MMA_RING_BYTES_LARGE_D
#define PD_MMA_RING_BYTES_LARGE_D (96 * 1024)
#endif
#ifndef PD_MMA_RING_BYTES_SPLIT_D256
#define PD_MMA_RING_BYTES_SPLIT_D256 (64 * 1024)
#endif
// per cache form at head_dim <= 128. The quantised stages carry a half (FP8)
// or a quarter (NVFP4) of BF16's bytes and their consumers are bound by the
// widening work, so more consumer warps beat more stages in flight: a 48 KB
// ring (three 16 KB FP8 stages) or a 40 KB one (four 10 KB NVFP4 stages) lets
// four CTAs share an SM (16 consumer warps instead of 12). Measured on the
// quantised batch: FP8 105.3 -> 93.3 us, NVFP4 108.7 -> 91.9 us per step.
#ifndef PD_MMA_RING_BYTES_FP8
#define PD_MMA_RING_BYTES_FP8 (48 * 1024)
#endif
#ifndef PD_MMA_RING_BYTES_NVFP4
#define PD_MMA_RING_BYTES_NVFP4 (40 * 1024)
#endif
template <int FMT>
constexpr int ring_bytes_small_d() {
  return FMT == PD_KV_NVFP4 ? PD_MMA_RING_BYTES_NVFP4
                            : (FMT == PD_KV_FP8_E4M3 ? PD_MMA_RING_BYTES_FP8
                                                     : PD_MMA_RING_BYTES_SMALL_D);
}
// CTAs per SM a partial kernel is compiled for (its register cap), from the
// shared memory one CTA takes: as many as fit an SM's 228 KB (one more KB
// reserved per CTA), at most four (4 x 160 threads x 96 registers fills the
// register file). With two q-head n-tiles (groups of 9-16) the accumulators
// need more registers than three CTAs leave, so those are compiled for two.
constexpr int partial_min_blocks(int smem_bytes, int nt) {
  return nt > 1 ? 2
                : ((228 * 1024) / (smem_bytes + 1024) > 4
                       ? 4
                       : ((228 * 1024) / (smem_bytes + 1024) < 1
                              ? 1
                              : (228 * 1024) / (smem_bytes + 1024)));
}

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
// Non-blocking probe of the same phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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
// Wait for the phase with the given parity to complete; false after limit_ns
// (default ~2 s).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// The same wait, which also gives up as soon as `abort_flag` (a shared-memory
// word another warp of the CTA sets when it stops) is non-zero. A limit of 0
// makes it a single non-blocking probe (a test's way to make waits run out).
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   const volatile int* abort_flag,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return mbar_test_wait(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag != 0 || global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// The same wait taken by a whole warp with one outcome for all its lanes
// (false if any lane ran out of time or `abort_flag` is set), so that the
// warp never splits on a wait that ends near its limit.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  return __all_sync(0xFFFFFFFFu, mbar_wait_or_abort(bar, parity, abort_flag, limit_ns));
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Four rows r0..r3 (any order, each may lie outside the tensor: zeros) of a
// 2-D tensor map whose box is one row high, from column x, landing one after
// another at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
// One NVFP4 stage of four 16-row pages for kv head g, by four lanes: lane 0
// gathers the K data slabs, 1 the V data slabs, 2 the K scale slabs, 3 the V
// scale slabs (maps as from encode_nvfp4_gather_map). pages[j] < 0 (no copy:
// outside the pool or past the key range) reads row oob_row, past the pool:
// zeros, with the same byte count. Lands as four pages of [16][D/2] data at
// kst / vst and four of [16][D/16] scales at + data_bytes_in_stage.
template <int D>
__device__ __forceinline__ void issue_nvfp4_gather(int lane, uint32_t kst, uint32_t vst,
                                                   uint32_t data_bytes_in_stage,
                                                   const CUtensorMap* tm_kd,
                                                   const CUtensorMap* tm_vd,
                                                   const CUtensorMap* tm_ks,
                                                   const CUtensorMap* tm_vs, int g,
                                                   int64_t page_data_bytes, const int* pages,
                                                   int oob_row, uint32_t bar) {
  constexpr int kSlabWords = 16 * (D / 2) / 4;    // a head's data slab in one page
  constexpr int kScaleWords = 16 * (D / 16) / 4;  // its scale slab
  if (lane >= 4) return;
  const int r0 = pages[0] >= 0 ? pages[0] : oob_row;
  const int r1 = pages[1] >= 0 ? pages[1] : oob_row;
  const int r2 = pages[2] >= 0 ? pages[2] : oob_row;
  const int r3 = pages[3] >= 0 ? pages[3] : oob_row;
  const bool scales = lane >= 2;
  const CUtensorMap* m = lane == 0 ? tm_kd : (lane == 1 ? tm_vd : (lane == 2 ? tm_ks : tm_vs));
  const uint32_t dst = ((lane & 1) ? vst : kst) + (scales ? data_bytes_in_stage : 0u);
  const int x = scales ? static_cast<int>(page_data_bytes / 4) + g * kScaleWords
                       : g * kSlabWords;
  tma_gather4(dst, m, x, r0, r1, r2, r3, bar);
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
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
// Host side: tensor maps.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
inline bool encode_cache_map(CUtensorMap* m, const void* base, int kv_dtype, int D, int hkv,
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

// 2-D map over an NVFP4 cache for page gathers: one row per page (row stride
// = the page stride), 32-bit elements across the page, box = box_bytes of one
// row. A gather at column x of four pages copies the same box_bytes-long
// section (a kv head's data slab or its scale slab) of each page.
inline bool encode_nvfp4_gather_map(CUtensorMap* m, const void* base, int64_t page_bytes,
                                    int64_t num_pages, int box_bytes) {
  auto fn = encode_fn();
  if (!fn || page_bytes % 16 != 0 || box_bytes % 16 != 0 || box_bytes / 4 > 256) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(page_bytes / 4),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(page_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / 4), 1u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE,
                         box_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                          : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

}  // namespace mma
}  // namespace pd
