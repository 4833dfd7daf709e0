// Paged prefill (chunked prefill) attention on mma.sync tensor-core tiles over
// the same paged cache the decode path reads, in every cache form.
//
// The pages name this unit beside decode: pegainfer issue 1008
// (`prefill_paged_launch` over the paged-KV view) and the AstrAI "csrc/tests"
// log (prefill kernels templated on the paged KV source, one causal offset,
// stride addressing for Q and O). Sequence b brings q_len_b query rows, its
// newest tokens: causal query i sits at position L_b - q_len_b + i and sees
// the keys up to itself; without causality every query sees all L_b keys. A
// window W keeps the last W keys before the query. The design is this
// library's own, for sm_103a:
//
//  * One CTA per (query tile, kv head, sequence) takes 64 (token, q head)
//    rows of the GQA group: 64 / G query tokens times the group's G heads,
//    16 rows per consumer warp, so each K/V byte a CTA loads serves every
//    head of the group. Tiles are numbered from the last one down: under
//    causality the last tiles see the most keys and start first.
//  * Warp 4 is the producer, as in the decode kernels: per 64-key tile it
//    looks up the pages in the block table (one int32 per page) and copies
//    each (page, kv head) slab of K and V into a ring stage (BF16: 3-D TMA
//    tensor copies with 128-byte swizzle; FP8: the same, unswizzled; NVFP4:
//    bulk copies of the data and scale slabs); stages complete on mbarrier
//    transaction counts and return through a second mbarrier. Every wait is
//    bounded, and the producer waits for every copy it issued before leaving.
//  * Warps 0-3 run the dense contraction on mma.sync m16n8k16 (fp32
//    accumulate), FlashAttention style: S = Q K^T with the warp's 16 rows on
//    M and 8-key n-tiles, K fragments by ldmatrix from the swizzled stage;
//    one online-softmax update per tile (row max over the four threads of a
//    row, exp2 with the scale folded into log2 units); P rebuilt from the S
//    accumulators as the A operand of O += P V, V fragments by
//    ldmatrix.trans. BF16 caches feed bf16 MMAs straight from the stage.
//    FP8 / NVFP4 stages are first widened, once per stage and by all four
//    warps together, into an f16 tile of the same swizzled layout: every
//    E4M3 value and every E2M1 x E4M3 product is an f16, so this is exact;
//    q enters the f16 MMAs multiplied by a power of two per row (its largest
//    magnitude into [2^14, 2^15)) and the factor, with the FP8 k_scale, is
//    folded into the row's score multiplier; the FP8 v_scale multiplies O at
//    the end.
//  * Keys outside a row's range score -inf. V rows that no row of the CTA may
//    read (before the CTA's first key, past its last, pages outside the pool)
//    are zeroed in the fragments, so whatever bytes sit in those stage rows
//    never reach the result.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "mma_common.cuh"
#include "pd_common.cuh"

namespace pd {
namespace {

using namespace ::pd::mma;

#ifndef PD_PREFILL_RING_BYTES
#define PD_PREFILL_RING_BYTES (96 * 1024)
#endif

template <int FMT, int D, int BS>
struct PCfg {
  static constexpr bool kQuant = FMT != PD_KV_BF16;   // widened to f16 before the MMAs
  static constexpr int kKT = 64;                      // keys per stage
  static constexpr int kBR = kKT < BS ? kKT : BS;     // rows per copy
  static constexpr int kNCopy = kKT / kBR;            // copies per stage and cache
  static constexpr int kCRB = 128;                    // bytes per swizzled chunk row
  static constexpr int kDCH = 2 * D / kCRB;           // 16-bit chunks per key row
  static constexpr int kCopyElems = kCRB / 2;         // box inner extent (bf16)
  // one key row of one head as stored in the cache (bytes) and a 16-bit
  // operand tile of the stage's keys (BF16: the stage itself; else the f16 tile)
  static constexpr int kRowBytes =
      FMT == PD_KV_BF16 ? 2 * D : (FMT == PD_KV_FP8_E4M3 ? D : D / 2);
  static constexpr int kOpCacheBytes = kKT * 2 * D;
  // NVFP4 stage: data [kKT][D/2] then scales [kKT][D/16]
  static constexpr int kDataBytes = kKT * kRowBytes;
  static constexpr int kScaleBytes = FMT == PD_KV_NVFP4 ? kKT * (D / 16) : 0;
  static constexpr int kCacheStageBytes =
      FMT == PD_KV_BF16 ? kOpCacheBytes : (kDataBytes + kScaleBytes + 1023) / 1024 * 1024;
  static constexpr int kStageBytes = 2 * kCacheStageBytes;
  static constexpr int kOpBytes = kQuant ? 2 * kOpCacheBytes : 0;  // the f16 K and V tiles
  static constexpr int kStagesRaw = (PD_PREFILL_RING_BYTES - kOpBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kOpOffset = kRingBytes;
  static constexpr int kBarOffset = kOpOffset + kOpBytes;
  // full[kStages], empty[kStages], the stages' bad-copy masks, the abort word
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + kStages * 4 + 16 + 1024;
  static constexpr uint32_t kCopyBytes =
      kBR * kRowBytes + (FMT == PD_KV_NVFP4 ? kBR * (D / 16) : 0);
  static constexpr int kKS = D / 16;  // k-steps of S = Q K^T
  static constexpr int kDT = D / 8;   // 8-wide head_dim tiles of O
  static_assert(kOpCacheBytes % 1024 == 0, "stages stay 1024-byte aligned for the swizzle");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
};

// Byte offset of (key, d) in a swizzled K or V stage: chunk-major rows of
// 128 bytes (64 bf16), keys 0..63 per chunk.
__device__ __forceinline__ uint32_t stage_off(int key, int d) {
  return swz128(static_cast<uint32_t>((d / 64) * (64 * 128) + key * 128 + (d % 64) * 2));
}

// One stage's K (or V) rows widened to f16 in the swizzled operand layout of
// the BF16 stage (chunk-major 128-byte rows, keys 0..63 per chunk), by the 128
// consumer threads together: thread t takes key t / 2, head_dim half t % 2.
// Exact: E4M3 values and E2M1 x E4M3 products are all f16 values.
template <int FMT, int D>
__device__ __forceinline__ void widen_stage(uint32_t raw, uint32_t op, int tid) {
  constexpr int kKT = 64;
  const int key = tid >> 1;
  const int e0 = (tid & 1) * (D / 2);
#pragma unroll
  for (int g8 = 0; g8 < D / 16; ++g8) {  // 8-element groups of this half row
    const int e = e0 + g8 * 8;
    uint32_t f[4];
    if constexpr (FMT == PD_KV_FP8_E4M3) {
      const uint2 w = lds64(raw + key * D + e);
      f[0] = e4m3x2_f16x2(w.x & 0xFFFFu);
      f[1] = e4m3x2_f16x2(w.x >> 16);
      f[2] = e4m3x2_f16x2(w.y & 0xFFFFu);
      f[3] = e4m3x2_f16x2(w.y >> 16);
    } else {
      const uint32_t w = lds32(raw + key * (D / 2) + e / 2);
      const uint32_t sc = lds_u8(raw + kKT * (D / 2) + key * (D / 16) + e / 16);
      const uint32_t s2 = e4m3x2_f16x2(sc | (sc << 8));
      uint32_t x[4];
      e2m1x8_f16x2(w, x);
#pragma unroll
      for (int k = 0; k < 4; ++k) f[k] = hmul2_u32(x[k], s2);
    }
    const uint32_t dst = op + (e / 64) * (kKT * 128) + swz128(key * 128 + ((e % 64) / 8) * 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(f[0]), "r"(f[1]),
                 "r"(f[2]), "r"(f[3])
                 : "memory");
  }
}

// (two CTAs per SM at head_dim <= 128; at 256 the O and Q fragments need the
// registers of one)
template <int FMT, int D, int BS>
__global__ void __launch_bounds__(kMmaThreads, D <= 128 ? 2 : 1)
    prefill_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  using C = PCfg<FMT, D, BS>;
  constexpr bool F16 = C::kQuant;
  // let a dependent grid be placed as this one drains (it waits for our
  // completion before reading anything we write)
  asm volatile("griddepcontrol.launch_dependents;");
  // a programmatic dependent of the previous work on the stream: nothing
  // global is read or written before that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tile = gridDim.x - 1 - blockIdx.x;  // the longest key ranges first
  const int G = a.group;
  const int TPC = a.tokens_per_cta;
  const int bs = a.block_size;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int r = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair

  // ---- the CTA's query tokens and the keys they may see ----
  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  const int L = a.seq_lens[b];
  const int tok0 = tile * TPC;
  // the grid covers max_q_len tokens: a longer sequence is flagged, not cut silently
  if (tile == static_cast<int>(gridDim.x) - 1 && q_len > static_cast<int>(gridDim.x) * TPC &&
      tid == 0)
    atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
  if (q_len <= 0 || tok0 >= q_len) return;
  if (L < q_len || L > a.max_blocks_per_seq * bs) {
    if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
    return;
  }
  const int tok1 = min(tok0 + TPC, q_len);
  const int pos_base = a.causal ? L - q_len : -1;  // position of token t: pos_base + t
  const int pos_first = a.causal ? pos_base + tok0 : L - 1;
  const int pos_last = a.causal ? pos_base + tok1 - 1 : L - 1;
  const int W = a.sliding_window;
  const int k_hi = pos_last + 1;                                   // keys [k_lo, k_hi)
  const int k_lo = (W > 0 && pos_first + 1 > W) ? pos_first + 1 - W : 0;
  const int t_base = (k_lo / bs) * bs;                             // page aligned
  const int ntiles = (k_hi - t_base + C::kKT - 1) / C::kKT;
  const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* ring = smem;
  const uint32_t op_k = smem_u32(smem + C::kOpOffset);  // f16 operand tiles (FP8 / NVFP4)
  const uint32_t op_v = op_k + C::kOpCacheBytes;
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
    if constexpr (FMT != PD_KV_NVFP4) {
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      }
    }
    const int64_t data_bytes = static_cast<int64_t>(bs) * a.num_kv_heads * (D / 2);
    const int64_t page_bytes = page_bytes_of(FMT, bs, a.num_kv_heads, D);
    // entries [cached_base, cached_base + 32) of the block-table row, one per lane
    int cached_base = -(1 << 30);
    int my_entry = -1;
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
        if (tt < k_hi) {
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
            const uint8_t* kp = static_cast<const uint8_t*>(a.k_cache) + my_page * page_bytes;
            const uint8_t* vp = static_cast<const uint8_t*>(a.v_cache) + my_page * page_bytes;
            constexpr uint32_t db = C::kBR * (D / 2);
            constexpr uint32_t sb = C::kBR * (D / 16);
            const uint32_t doff = j * db;
            const uint32_t soff = C::kDataBytes + j * sb;
            bulk_load(kst + doff, kp + line * (D / 2), db, fb);
            bulk_load(vst + doff, vp + line * (D / 2), db, fb);
            bulk_load(kst + soff, kp + data_bytes + line * (D / 16), sb, fb);
            bulk_load(vst + soff, vp + data_bytes + line * (D / 16), sb, fb);
          } else if constexpr (FMT == PD_KV_FP8_E4M3) {
            // one unswizzled box of kBR rows x D bytes: [key][D] in the stage
            const int z = my_page * bs + row0;
            const uint32_t off = j * (C::kBR * D);
            tma_load_3d(kst + off, &tm_k, 0, g, z, fb);
            tma_load_3d(vst + off, &tm_v, 0, g, z, fb);
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
  // rows m0 = 16 warp + r and m1 = m0 + 8 of the CTA's 64: token m / G, head m % G
  int rpos[2], rlo[2];
  bool rvalid[2];
  const uint16_t* qrow[2];
  uint16_t* orow[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int m = warp * 16 + r + 8 * hh;
    const int t = tok0 + m / G;
    rvalid[hh] = (m / G) < TPC && t < tok1;
    const int tt = rvalid[hh] ? t : tok0;
    const int qh = g * G + m % G;
    rpos[hh] = a.causal ? pos_base + tt : L - 1;
    rlo[hh] = (W > 0 && rpos[hh] + 1 > W) ? rpos[hh] + 1 - W : 0;
    if (!rvalid[hh]) rpos[hh] = -1;  // sees no key
    qrow[hh] = a.q + static_cast<int64_t>(q0 + tt) * a.q_stride + static_cast<int64_t>(qh) * D;
    orow[hh] = a.out + static_cast<int64_t>(q0 + tt) * a.out_stride + static_cast<int64_t>(qh) * D;
  }
  // Q as A fragments: a0 (row m0, d 2c..), a1 (m1), a2 (m0, d 8+2c..), a3 (m1)
  uint32_t qa[C::kKS][4];
#pragma unroll
  for (int ks = 0; ks < C::kKS; ++ks) {
    const int d = ks * 16 + 2 * c;
    qa[ks][0] = rvalid[0] ? *reinterpret_cast<const uint32_t*>(qrow[0] + d) : 0u;
    qa[ks][1] = rvalid[1] ? *reinterpret_cast<const uint32_t*>(qrow[1] + d) : 0u;
    qa[ks][2] = rvalid[0] ? *reinterpret_cast<const uint32_t*>(qrow[0] + d + 8) : 0u;
    qa[ks][3] = rvalid[1] ? *reinterpret_cast<const uint32_t*>(qrow[1] + d + 8) : 0u;
  }
  // score multiplier (log2 units) of rows m0, m1
  float sl2[2] = {a.scale_log2, a.scale_log2};
  if constexpr (F16) {
    // q into f16 times a power of two per row, max |q| of the row in
    // [2^14, 2^15) (exact: f16 holds bf16's 8 significant bits); the row's
    // four threads (c = 0..3) hold all of its head_dim
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mq = 0.0f;
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks)
#pragma unroll
        for (int e = hh; e < 4; e += 2)
          mq = fmaxf(mq, fmaxf(fabsf(bf16_lo(qa[ks][e])), fabsf(bf16_hi(qa[ks][e]))));
      mq = fmaxf(mq, __shfl_xor_sync(0xFFFFFFFFu, mq, 1));
      mq = fmaxf(mq, __shfl_xor_sync(0xFFFFFFFFu, mq, 2));
      const float qdown = exp2i(14 - ilog2f(mq));
      sl2[hh] = a.scale_log2 * (FMT == PD_KV_FP8_E4M3 ? a.k_scale : 1.0f) *
                exp2i(ilog2f(mq) - 14);
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks)
#pragma unroll
        for (int e = hh; e < 4; e += 2)
          qa[ks][e] = pack_f16x2(bf16_lo(qa[ks][e]) * qdown, bf16_hi(qa[ks][e]) * qdown);
    }
  }
  const float vmul = FMT == PD_KV_FP8_E4M3 ? a.v_scale : 1.0f;
  float acc[C::kDT][4];
#pragma unroll
  for (int dt = 0; dt < C::kDT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row this lane addresses

  bool failed = false;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::kStages;
    bool ok = warp_wait(smem_u32(&full_bar[st]), (i / C::kStages) & 1, abort_s);
    // FP8 / NVFP4: the four warps widen the stage together and meet at named
    // barriers, so they agree on every wait's outcome first
    if constexpr (F16) ok = consumers_vote(ok);
    if (!ok) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      *abort_s = 1;
      failed = true;
      break;
    }
    uint32_t kst = smem_u32(ring + st * C::kStageBytes);
    uint32_t vst = kst + C::kCacheStageBytes;
    const uint32_t bad = bad_copies[st];
    const int t0 = t_base + i * C::kKT;
    if constexpr (F16) {
      consumers_sync();  // every warp is done with the previous tile's f16 operands
      widen_stage<FMT, D>(kst, op_k, tid);
      widen_stage<FMT, D>(vst, op_v, tid);
      consumers_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // the raw stage is free
      kst = op_k;
      vst = op_v;
    }

    // ---- S = Q K^T: 16 rows x 64 keys, eight n-tiles of 8 keys ----
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < C::kKS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t kb[4];
        ldsm_x4(kst + stage_off((2 * np + (mi >> 1)) * 8 + ri, ks * 16 + (mi & 1) * 8), kb);
        mma16816<F16>(s[2 * np], qa[ks], kb[0], kb[1]);
        mma16816<F16>(s[2 * np + 1], qa[ks], kb[2], kb[3]);
      }
    }

    // ---- mask, scale, one online-softmax update per row ----
    // element e of n-tile nt: row m0 (e < 2) or m1, key t0 + 8 nt + 2c + (e & 1)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = e >> 1;
        const int kk = nt * 8 + 2 * c + (e & 1);
        const int key = t0 + kk;
        const bool okk = key >= rlo[hh] && key <= rpos[hh] && !((bad >> (kk / C::kBR)) & 1u);
        s[nt][e] = okk ? s[nt][e] * sl2[hh] : -INFINITY;
        mx[hh] = fmaxf(mx[hh], s[nt][e]);
      }
    float alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xFFFFFFFFu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xFFFFFFFFu, mx[hh], 2));
      const float mn = fmaxf(m_run[hh], mx[hh]);
      alpha[hh] = (mn == -INFINITY) ? 1.0f : ex2(m_run[hh] - mn);
      m_run[hh] = mn;
    }
    float ls[2] = {0.0f, 0.0f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = e >> 1;
        s[nt][e] = (m_run[hh] == -INFINITY) ? 0.0f : ex2(s[nt][e] - m_run[hh]);
        ls[hh] += s[nt][e];
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) l_run[hh] = l_run[hh] * alpha[hh] + ls[hh];
#pragma unroll
    for (int dt = 0; dt < C::kDT; ++dt) {
      acc[dt][0] *= alpha[0];
      acc[dt][1] *= alpha[0];
      acc[dt][2] *= alpha[1];
      acc[dt][3] *= alpha[1];
    }

    // ---- O += P V, 16 keys per k-step ----
    // V rows no row of the CTA may read are zeroed (stale stage bytes)
    const bool ragged = t0 < k_lo || t0 + C::kKT > k_hi || bad != 0u;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      uint32_t pa[4];
      if constexpr (F16) {
        pa[0] = pack_f16x2(s[2 * kb][0], s[2 * kb][1]);
        pa[1] = pack_f16x2(s[2 * kb][2], s[2 * kb][3]);
        pa[2] = pack_f16x2(s[2 * kb + 1][0], s[2 * kb + 1][1]);
        pa[3] = pack_f16x2(s[2 * kb + 1][2], s[2 * kb + 1][3]);
      } else {
        pa[0] = pack_bf16x2(s[2 * kb][0], s[2 * kb][1]);
        pa[1] = pack_bf16x2(s[2 * kb][2], s[2 * kb][3]);
        pa[2] = pack_bf16x2(s[2 * kb + 1][0], s[2 * kb + 1][1]);
        pa[3] = pack_bf16x2(s[2 * kb + 1][2], s[2 * kb + 1][3]);
      }
      uint32_t keep_lo = 0xFFFFFFFFu, keep_hi = 0xFFFFFFFFu;
      if (ragged) {
        auto key_ok = [&](int kk) {
          const int key = t0 + kk;
          return key >= k_lo && key < k_hi && !((bad >> (kk / C::kBR)) & 1u);
        };
        const int k0 = kb * 16 + 2 * c;
        keep_lo = (key_ok(k0) ? 0x0000FFFFu : 0u) | (key_ok(k0 + 1) ? 0xFFFF0000u : 0u);
        keep_hi = (key_ok(k0 + 8) ? 0x0000FFFFu : 0u) | (key_ok(k0 + 9) ? 0xFFFF0000u : 0u);
      }
#pragma unroll
      for (int dp = 0; dp < C::kDT / 2; ++dp) {
        uint32_t vb[4];
        ldsm_x4_trans(vst + stage_off((kb * 16 + (mi & 1) * 8 + ri), (2 * dp + (mi >> 1)) * 8), vb);
        vb[0] &= keep_lo;
        vb[1] &= keep_hi;
        vb[2] &= keep_lo;
        vb[3] &= keep_hi;
        mma16816<F16>(acc[2 * dp], pa, vb[0], vb[1]);
        mma16816<F16>(acc[2 * dp + 1], pa, vb[2], vb[3]);
      }
    }
    if constexpr (!F16) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
  }
  if (failed) return;

  // ---- out = O / l, bf16 ----
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xFFFFFFFFu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xFFFFFFFFu, l_run[hh], 2);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (!rvalid[hh]) continue;
    const float inv = vmul / fmaxf(l_run[hh], 1e-20f);
#pragma unroll
    for (int dt = 0; dt < C::kDT; ++dt) {
      const uint32_t v = pack_bf16x2(acc[dt][2 * hh] * inv, acc[dt][2 * hh + 1] * inv);
      *reinterpret_cast<uint32_t*>(orow[hh] + dt * 8 + 2 * c) = v;
    }
  }
}

template <int FMT, int D, int BS>
cudaError_t launch_prefill_cfg(const PrefillArgs& a, const void* kc, const void* vc,
                               int max_q_len, cudaStream_t st) {
  using C = PCfg<FMT, D, BS>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  const int64_t rows = a.num_blocks * a.block_size;
  if constexpr (FMT == PD_KV_BF16) {
    if (!encode_cache_map(&tk, kc, PD_KV_BF16, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          true) ||
        !encode_cache_map(&tv, vc, PD_KV_BF16, D, a.num_kv_heads, rows, C::kCopyElems, C::kBR,
                          true))
      return cudaErrorInvalidValue;
  } else if constexpr (FMT == PD_KV_FP8_E4M3) {
    // whole D-byte rows, unswizzled (the consumers widen them element-wise)
    if (!encode_cache_map(&tk, kc, PD_KV_FP8_E4M3, D, a.num_kv_heads, rows, D, C::kBR, false) ||
        !encode_cache_map(&tv, vc, PD_KV_FP8_E4M3, D, a.num_kv_heads, rows, D, C::kBR, false))
      return cudaErrorInvalidValue;
  }
  auto kern = prefill_mma_kernel<FMT, D, BS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};  // per device; setting it twice is harmless
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int tiles = (max_q_len + a.tokens_per_cta - 1) / a.tokens_per_cta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, a.num_kv_heads, a.num_seqs);
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

template <int FMT>
cudaError_t launch_prefill_fmt(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                               int head_dim, int max_q_len, cudaStream_t st) {
  const bool bs16 = a.block_size == 16;
  switch (head_dim) {
    case 64:
      return bs16 ? launch_prefill_cfg<FMT, 64, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_prefill_cfg<FMT, 64, 32>(a, k_cache, v_cache, max_q_len, st);
    case 128:
      return bs16 ? launch_prefill_cfg<FMT, 128, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_prefill_cfg<FMT, 128, 32>(a, k_cache, v_cache, max_q_len, st);
    case 256:
      return bs16 ? launch_prefill_cfg<FMT, 256, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_prefill_cfg<FMT, 256, 32>(a, k_cache, v_cache, max_q_len, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                           int head_dim, int kv_dtype, int max_q_len, cudaStream_t st) {
  if (a.num_seqs == 0 || max_q_len == 0) return cudaSuccess;
  switch (kv_dtype) {
    case PD_KV_BF16:
      return launch_prefill_fmt<PD_KV_BF16>(a, k_cache, v_cache, head_dim, max_q_len, st);
    case PD_KV_FP8_E4M3:
      return launch_prefill_fmt<PD_KV_FP8_E4M3>(a, k_cache, v_cache, head_dim, max_q_len, st);
    default:
      return launch_prefill_fmt<PD_KV_NVFP4>(a, k_cache, v_cache, head_dim, max_q_len, st);
  }
}

}  // namespace pd
