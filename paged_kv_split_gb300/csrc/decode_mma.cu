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

#include "mma_common.cuh"
#include "mma_tile.cuh"
#include "pd_common.cuh"

// Cfg<> defines every layout constant for every form; NVFP4 ignores some.
#pragma nv_diag_suppress 177

namespace pd {
namespace {

using namespace ::pd::mma;

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
      (kDSplit == 1 ? ring_bytes_small_d<FMT>()
                    : (D == 256 ? PD_MMA_RING_BYTES_SPLIT_D256 : PD_MMA_RING_BYTES_LARGE_D)) /
      kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  // cross-warp score sums (head_dim split): 2 buffers x 4 warps x m-tiles x 32 lanes x 4*NT
  static constexpr int kRedBytes = kDSplit == 4 ? 2 * 4 * kMT * 32 * 4 * NT * 4 : 0;
  static constexpr int kMergeBytes = kDSplit == 1 ? 4 * (kDS * 8 * NT + 2 * 8 * NT) * 4 : 0;
  static_assert(kMergeBytes <= kRingBytes, "the end-of-CTA merge reuses the ring");
  static constexpr int kQMaxBytes = kDSplit == 4 ? 2 * 4 * 8 * 4 : 0;  // [NT][warp][8] floats
  static constexpr int kBarOffset = kRingBytes + kRedBytes + kQMaxBytes;
  // full[kStages], empty[kStages], the stages' bad-copy masks, the abort word
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + kStages * 4 + 16 + 1024;
  // per copy and cache: bytes landed by TMA
  static constexpr uint32_t kCopyBytes =
      kBR * kRowBytes + (FMT == PD_KV_NVFP4 ? kBR * (D / 16) : 0);
  // NVFP4 with 16-row pages and 64-key stages: one gather of the stage's four
  // pages per cache and section (data slab, scale slab) instead of four bulk
  // copies each, so a 9 KB stage takes 4 copy operations instead of 16
  static constexpr bool kGather = FMT == PD_KV_NVFP4 && BS == 16 && kDSplit == 1;
  static_assert(!kGather || kNCopy == 4, "a gather covers exactly four pages");
};

template <int FMT, int D, int NT, int BS>
__global__ void __launch_bounds__(kMmaThreads,
                                  partial_min_blocks(Cfg<FMT, D, NT, BS>::kSmemBytes, NT))
    partial_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs, const DecodeArgs a) {
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
    if constexpr (FMT != PD_KV_NVFP4 || C::kGather) {
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      }
      if constexpr (C::kGather) {
        if (lane == 1) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_ks)) : "memory");
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_vs)) : "memory");
        }
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
      uint16_t* o = a.out + static_cast<int64_t>(b) * a.out_stride + g * G * D;
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
  // set by a warp that stops early: the others stop waiting on it
  volatile int* abort_s = reinterpret_cast<volatile int*>(bad_copies + C::kStages);

  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kConsumerWarps);
    }
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // =========================== producer warp ===============================
  if (warp == kConsumerWarps) {
    // entries [cached_base, cached_base + 32) of the block-table row, one per lane
    int cached_base = a.sliding_window == 0 ? s * a.chunk : -(1 << 30);
    int my_entry = spec_entry;
    int i = 0;  // tiles issued
    for (; i < ntiles; ++i) {
      const int st = i % C::kStages;
      // a stage is re-armed only after all four consumer warps have handed it
      // back, which they do only after its previous copies landed
      if (i >= C::kStages &&
          !warp_wait(smem_u32(&empty_bar[st]), ((i / C::kStages) - 1) & 1, abort_s)) {
        if (lane == 0 && *abort_s == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
        *abort_s = 1;
        break;  // the consumers stopped, or this wait ran out: issue nothing more
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
      if constexpr (C::kGather) {
        if (bytes != 0) bytes = 2u * C::kNCopy * C::kCopyBytes;  // pages past the pool land zeros
      }
      const uint32_t fb = smem_u32(&full_bar[st]);
      if (lane == 0) {
        if (bad) atomicOr(a.flags, PD_DEV_BAD_PAGE);
        bad_copies[st] = bad;
        mbar_arrive_expect_tx(fb, bytes);
      }
      __syncwarp();
      // one lane per page issues that page's copies, in parallel (NVFP4 with
      // 16-row pages: four lanes each gather one section of all four pages)
      if constexpr (C::kGather) {
        if (bytes != 0) {
          const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
          issue_nvfp4_gather<D>(lane, kst, kst + C::kCacheStageBytes, C::kDataBytes, &tm_k, &tm_v,
                                &tm_ks, &tm_vs, g, a.data_bytes, pages,
                                static_cast<int>(a.num_blocks), fb);
        }
      } else {
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
    // every copy issued lands before the CTA can end (consumers that gave up
    // no longer wait for them)
    for (int t = max(0, i - C::kStages); t < i; ++t)
      (void)mbar_wait(smem_u32(&full_bar[t % C::kStages]), (t / C::kStages) & 1);
    return;
  }

  // =========================== consumer warps ==============================
  const int d0 = C::kDSplit == 4 ? warp * C::kDS : 0;  // this warp's head_dim slice

  const ThreadPlace tp{warp, lane, r, c, d0};
  TileState<C, NT> ts;
  load_q_fragments<FMT, D, NT>(ts, a.q + static_cast<int64_t>(b) * a.q_stride + g * G * D, G,
                               a.scale_log2, a.k_scale, tp, qmax_s);
  reset_state(ts);
  auto& acc = ts.acc;
  auto& m_run = ts.m_run;
  auto& l_run = ts.l_run;

  bool failed = false;
  int red_buf = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::kStages;
    // after one failed wait, stop waiting (bounded total time) and stop handing
    // stages back, so that the producer re-arms none whose copies may still be
    // landing; results are then discarded, but every named barrier is reached
    if (!failed && !warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s,
                              a.consumer_wait_ns)) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      *abort_s = 1;
      failed = true;
    }
    const uint32_t kst = smem_u32(ring + st * C::kStageBytes);
    const uint32_t vst = kst + C::kCacheStageBytes;
    const uint32_t bad = bad_copies[st];
    const int t0 = t_base + i * C::kKT;

    consume_tile<FMT, D, NT>(ts, StageView{kst, vst, t0, t_begin, t_end, bad}, tp, red, red_buf);
    if constexpr (C::kDSplit == 4) red_buf ^= 1;
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(smem_u32(&empty_bar[st]));
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

  const int64_t orow0 = static_cast<int64_t>(b) * a.out_stride + g * G * D;  // out row of head 0
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

template <int FMT, int D, int NT, int BS>
cudaError_t launch_mma_cfg(const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<FMT, D, NT, BS>;
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
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, tks, tvs, a);
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
    smem = head_dim <= 128   ? Cfg<PD_KV_BF16, 128, 1, 16>::kSmemBytes
           : head_dim == 256 ? Cfg<PD_KV_BF16, 256, 1, 16>::kSmemBytes
                             : Cfg<PD_KV_BF16, 512, 1, 16>::kSmemBytes;
  } else if (kv_dtype == PD_KV_FP8_E4M3) {
    smem = head_dim <= 128   ? Cfg<PD_KV_FP8_E4M3, 128, 1, 16>::kSmemBytes
           : head_dim == 256 ? Cfg<PD_KV_FP8_E4M3, 256, 1, 16>::kSmemBytes
                             : Cfg<PD_KV_FP8_E4M3, 512, 1, 16>::kSmemBytes;
  } else {
    smem = head_dim <= 128   ? Cfg<PD_KV_NVFP4, 128, 1, 16>::kSmemBytes
           : head_dim == 256 ? Cfg<PD_KV_NVFP4, 256, 1, 16>::kSmemBytes
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
