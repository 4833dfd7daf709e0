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
//    ends with an error instead of hanging. A warp that gives up raises the
//    CTA's abort word, which every other wait polls; the producer then issues
//    nothing more and waits for the copies it already issued before leaving.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "mma_common.cuh"
#include "mma_tile.cuh"
#include "pd_common.cuh"

// Cfg<> defines every layout constant for every form; NVFP4 ignores some.
#pragma nv_diag_suppress 177

namespace pd {
namespace {

using namespace ::pd::mma;

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
      (kDSplit == 1 ? ring_bytes_small_d<FMT>() : PD_MMA_RING_BYTES_LARGE_D) / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  // cross-warp score sums (head_dim split): 2 buffers x 4 warps x m-tiles x 32 lanes x 4*NT
  static constexpr int kRedBytes = kDSplit == 4 ? 2 * 4 * kMT * 32 * 4 * NT * 4 : 0;
  static constexpr int kQMaxBytes = kDSplit == 4 ? NT * 4 * 8 * 4 : 0;  // [NT][warp][8] floats
  static constexpr int kHW = 8 * NT;                        // q-head columns of the tiles
  static constexpr int kMStride = D + 4;                    // floats per merge-slice row
  // the four warps' unscaled O of a piece fit the piece's held last stage (as
  // [warp][head][D] floats) for every group this instantiation serves: then
  // the merge needs no slice of its own
  static constexpr bool kMergeInStage = 4 * kHW * D * 4 <= kStageBytes;
  // end-of-item merge (head_dim <= 128): a [kHW][D+4] slice (unless the held
  // stage takes the merge), per-warp m and l (two buffers, by item parity),
  // and the merged m and l of each column
  static constexpr int kMergeBytes =
      kDSplit == 1 ? ((kMergeInStage ? 0 : kHW * kMStride) + 2 * 2 * 4 * kHW + 2 * kHW) * 4 : 0;
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
  // NVFP4 with 16-row pages and 64-key stages: one gather of the stage's four
  // pages per cache and section (data slab, scale slab) instead of four bulk
  // copies each, so a 9 KB stage takes 4 copy operations instead of 16
  static constexpr bool kGather = FMT == PD_KV_NVFP4 && BS == 16 && kDSplit == 1;
  static_assert(!kGather || kNCopy == 4, "a gather covers exactly four pages");
  // dynamic shared memory for a GQA group of G heads (q slots of G rows),
  // with 1 KB of slack for aligning the ring to 1024 bytes
  static constexpr int smem_bytes(int G) { return kQOffset + kQSlots * G * D * 2 + 1024; }
};

// Consumer-warp barrier on an mbarrier (one arrival per warp, bounded wait),
// so that a stalled peer ends in an error instead of a hang.
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
__global__ void __launch_bounds__(kMmaThreads,
                                  partial_min_blocks(Cfg<FMT, D, NT, BS>::smem_bytes(8 * NT), NT))
    partial_balanced_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs, const DecodeArgs a) {
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
  float* mslice = reinterpret_cast<float*>(smem + C::kMergeOffset);  // [kHW][D+4], if any
  float* mrec = mslice + (C::kMergeInStage ? 0 : C::kHW * C::kMStride);  // [2][4][kHW]
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
  if constexpr (FMT != PD_KV_NVFP4 || C::kGather) {
    if (tid == kConsumerWarps * 32) {  // the tensor maps are kernel parameters
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      if constexpr (C::kGather) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_ks)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_vs)) : "memory");
      }
    }
  }
  __syncthreads();
  // Launched as a programmatic dependent of whatever came before on the
  // stream (the previous step's combine, say): nothing global is read or
  // written before that grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // =========================== producer warp ===============================
  if (warp == kConsumerWarps) {
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
          if constexpr (C::kGather) {
            if (bytes != 0) bytes = 2u * C::kNCopy * C::kCopyBytes;  // pages past the pool land zeros
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
          if constexpr (C::kGather) {
            if (bytes > (j == 0 ? q_bytes : 0u)) {
              const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
              issue_nvfp4_gather<D>(lane, kst, kst + C::kCacheStageBytes, C::kDataBytes, &tm_k,
                                    &tm_v, &tm_ks, &tm_vs, g, a.data_bytes, pages,
                                    static_cast<int>(a.num_blocks), fb);
            }
          } else {
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
    }
    // every copy issued lands before the block can exit (consumers that gave
    // up no longer wait for them)
    for (int t = max(0, i - C::kStages); t < i; ++t)
      (void)mbar_wait(smem_u32(&full_bar[t % C::kStages]), (t / C::kStages) & 1);
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

  const ThreadPlace tp{warp, lane, r, c, d0};
  int i = 0;  // tiles consumed
  int red_buf = 0;
  int ip = 0;  // item parity (merge buffers)
  bool aborted = false;
  while (!aborted) {
    int st = i % C::kStages;
    {
      bool ok = warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s,
                          a.consumer_wait_ns);
      // head_dim split: the warps meet at named barriers every tile, so they
      // must agree on every wait's outcome before reading the stage record
      if constexpr (C::kDSplit == 4) ok = consumers_vote(ok);
      if (!ok) {
        if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
        *abort_s = 1;
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

    // ---- q fragments of the piece's GQA group, from its q slot ----
    TileState<C, NT> ts;
    load_q_fragments<FMT, D, NT>(ts, reinterpret_cast<const uint16_t*>(qslots + qslot * q_bytes),
                                 G, a.scale_log2, a.k_scale, tp, qmax_s);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&qempty_bar[qslot]));

    // ---- running state of the piece ----
    reset_state(ts);
    auto& acc = ts.acc;
    auto& m_run = ts.m_run;
    auto& l_run = ts.l_run;

    // ---- the item's tiles ----
    while (true) {
    const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
    const uint32_t vst = kst + C::kCacheStageBytes;
    const uint32_t bad = meta[st].bad;
    const int t0 = meta[st].t0;
    consume_tile<FMT, D, NT>(ts, StageView{kst, vst, t0, t_begin, t_end, bad}, tp, red, red_buf);
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
      bool ok = warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s,
                          a.consumer_wait_ns);
      if constexpr (C::kDSplit == 4) ok = consumers_vote(ok);
      if (!ok) {
        if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
        *abort_s = 1;
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
    const int64_t orow0 = static_cast<int64_t>(b) * a.out_stride + g * G * D;  // head 0's row
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
      // padded rows (conflict-free fragment stores) where they fit the stage
      const int ostride = 4 * G * (D + 4) * 4 <= C::kStageBytes ? D + 4 : D;
      if (C::kMergeInStage || 4 * G * ostride * 4 <= C::kStageBytes) {
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

template <int FMT, int D, int NT, int BS>
cudaError_t launch_bal_cfg(const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<FMT, D, NT, BS>;
  const int smem = C::smem_bytes(a.group);
  CUtensorMap tk, tv, tks, tvs;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  std::memset(&tks, 0, sizeof(tks));
  std::memset(&tvs, 0, sizeof(tvs));
  if constexpr (FMT != PD_KV_NVFP4) {
    const int64_t rows = a.num_blocks * a.block_size;
    if (!encode_cache_map(&tk, a.k_cache, FMT, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          C::kSwizzle) ||
        !encode_cache_map(&tv, a.v_cache, FMT, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          C::kSwizzle))
      return cudaErrorInvalidValue;
  } else if constexpr (C::kGather) {
    // page gathers: data slabs ([16][D/2] bytes of a head) and scale slabs
    // ([16][D/16]) of whole pages
    constexpr int kSlab = 16 * (D / 2), kScales = 16 * (D / 16);
    if (!encode_nvfp4_gather_map(&tk, a.k_cache, a.page_bytes, a.num_blocks, kSlab) ||
        !encode_nvfp4_gather_map(&tv, a.v_cache, a.page_bytes, a.num_blocks, kSlab) ||
        !encode_nvfp4_gather_map(&tks, a.k_cache, a.page_bytes, a.num_blocks, kScales) ||
        !encode_nvfp4_gather_map(&tvs, a.v_cache, a.page_bytes, a.num_blocks, kScales))
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
  // A programmatic dependent of the previous work on the stream: the grid is
  // placed, and its barriers set up, while the previous combine grid drains.
  // The plan gives every CTA an equal share on the assumption that all of
  // them start together; that holds because the combine lets its dependents
  // launch only as its CTAs finish, so no combine CTA still holds the
  // registers a third partial CTA of an SM needs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan_num_ctas);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, tks, tvs, a);
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
