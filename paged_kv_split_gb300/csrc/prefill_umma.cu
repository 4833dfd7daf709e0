// Paged prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// TMEM) over the BF16 paged cache, head_dim 256 (one 128-row query tile per
// CTA: O takes 256 TMEM columns, so two tiles do not fit; head_dim 64 and 128
// run two tiles per CTA in prefill_pair.cu). Same semantics and interface as
// the mma.sync kernel in prefill_mma.cu (which stays as a cross-check):
// pegainfer issue 1008 (`prefill_paged_launch`), AstrAI "csrc/tests" log
// (causal offset, stride addressing). Design, for sm_103a:
//
//  * One CTA per (query tile, kv head, sequence) owns 128 (token, q head)
//    rows: 128 / G query tokens times the GQA group's G heads, so every K/V
//    byte it loads serves the whole group. Tiles run from the last one down
//    (under causality the last tiles see the most keys).
//  * Warp 8 (producer) copies 64-key K and V tiles of the kv head into a ring
//    with 3-D TMA tensor copies (128-byte swizzle), one block-table lookup per
//    page; copies it skips (pages outside the pool, rows past the CTA's keys)
//    are issued at a row past the pool, which TMA fills with zeros.
//  * Warp 9 allocates 256 TMEM columns and one of its threads issues the MMAs:
//    S_j = Q K_j^T (M = 128 rows, N = 64 keys, K = head_dim; Q and K K-major in
//    shared memory) into one of two TMEM buffers, so S_{j+1} runs while the
//    softmax of tile j does; O += P_j V_j (N = head_dim; P K-major in shared
//    memory, V MN-major straight from the stage) into a TMEM accumulator.
//    tcgen05.commit signals each result on an mbarrier.
//  * Warps 0-7 run the softmax, two threads per row: warp w owns rows
//    32 (w % 4) .. +31 (TMEM lanes of its warp's quarter) and key half w / 4
//    of each 64-key tile. Per tile a thread reads its 32 scores with
//    tcgen05.ld, masks them (causal position, window, pages outside the pool)
//    with one 32-bit valid-key word, swaps its half-row max with its partner
//    through shared memory (one named barrier per tile), writes its P slice
//    as bf16 into the swizzled A-operand tile, and the pair rescales O in TMEM
//    only when the tile max passes the reference max by more than 2^8 (P stays
//    <= 256; the result is the same up to rounding). V rows of keys no row of
//    the CTA may read are zeroed first, so stale stage bytes never meet a zero
//    weight. The epilogue adds the two partial row sums and writes O / l.
//  * Every mbarrier wait is bounded (2 s): on time-out the CTA raises
//    PD_DEV_TIMEOUT, stops issuing work, waits (bounded) for what it issued,
//    frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "mma_common.cuh"
#include "pd_common.cuh"
#include "umma_common.cuh"

namespace pd {
namespace {

using namespace ::pd::mma;
using namespace ::pd::umma;

// K/V stages of the ring: the copies of a tile must be issued several tiles
// ahead of its MMAs to cover the loaded memory latency
#ifndef PD_UMMA_PREFILL_STAGES
#define PD_UMMA_PREFILL_STAGES 0  // 0: five stages at head_dim 128, four at 64
#endif
// CTAs per SM the kernel is compiled for (its register cap)
#ifndef PD_UMMA_PREFILL_MIN_BLOCKS
#define PD_UMMA_PREFILL_MIN_BLOCKS 1
#endif
// The running max that P is taken against moves only when a row's tile max
// exceeds it by more than this (log2 units): P <= 2^8 in bf16, and O and l
// are rescaled in TMEM a few times per row instead of nearly every tile.
constexpr float kRescaleLog2 = 8.0f;

// warps 0-7 softmax (warp w: rows 32 (w % 4) .. +31, key half w / 4),
// warp 8 producer, warp 9 MMA issuer
constexpr int kSoftWarps = 8;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kUmmaThreads = 10 * 32;
constexpr int kRowsU = 128;           // (token, q head) rows per CTA = UMMA M
// TMEM columns: S0 [0, 64), S1 [64, 128), O [128, 128 + D), rounded up to a
// power of two (head_dim 256 takes all 512 columns of the SM)
template <int D>
constexpr int tmem_cols() { return D <= 128 ? 256 : 512; }

template <int D, int BS>
struct UCfg {
  static constexpr int kKT = 64;                      // keys per stage (UMMA N of S)
  static constexpr int kBR = kKT < BS ? kKT : BS;     // rows per copy
  static constexpr int kNCopy = kKT / kBR;
  static constexpr int kDCH = D / 64;                 // 64-element (128-byte) chunks per row
  static constexpr int kQBytes = kDCH * kRowsU * 128;  // Q tile, chunk-major
  static constexpr int kPBytes = kRowsU * 128;         // P tile: 128 rows x 64 keys bf16
  static constexpr int kCacheStageBytes = kKT * 2 * D;
  static constexpr int kStageBytes = 2 * kCacheStageBytes;
  // five stages at head_dim 128, four at 64; at 256 a stage is 64 KB and two
  // fit beside the 64 KB Q tile
  static constexpr int kStages =
      PD_UMMA_PREFILL_STAGES > 0 ? PD_UMMA_PREFILL_STAGES
                                 : (D == 128 ? 5 : (D == 64 ? 4 : 2));
  static constexpr int kQOff = 0;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kRingOff = kPOff + kPBytes;
  static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
  // kv_full[S], kv_empty[S], s_full[2], s_free[2], p_full, o_done, final
  static constexpr int kNumBars = 2 * kStages + 7;
  // the two threads of a row swap their half-row max (two buffers by tile
  // parity) and, at the end, their partial row sums
  static constexpr int kXOff = kBarOff + kNumBars * 8;       // float [2][2][128]
  static constexpr int kLOff = kXOff + 2 * 2 * kRowsU * 4;   // float [2][128]
  static constexpr int kBadOff = kLOff + 2 * kRowsU * 4;
  static constexpr int kHolderOff = kBadOff + kStages * 4;
  // no alignment slack (it would cost a stage): the kernel checks that
  // dynamic shared memory starts on a 1024-byte boundary
  static constexpr int kSmemBytes = kHolderOff + 16;
  static constexpr uint32_t kCopyBytes = kBR * 2 * D;
  static constexpr int kKS = D / 16;  // K steps of S
  static_assert(kCacheStageBytes % 1024 == 0 && kQBytes % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
};

template <int D, int BS>
__global__ void __launch_bounds__(kUmmaThreads, PD_UMMA_PREFILL_MIN_BLOCKS)
    prefill_umma_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  using C = UCfg<D, BS>;
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tile = gridDim.x - 1 - blockIdx.x;  // the longest key ranges first
  const int G = a.group;
  const int TPC = a.tokens_per_cta;  // 128 / G
  const int bs = a.block_size;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- the CTA's query tokens and the keys they may see ----
  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  const int L = a.seq_lens[b];
  const int tok0 = tile * TPC;
  if (tile == static_cast<int>(gridDim.x) - 1 && q_len > static_cast<int>(gridDim.x) * TPC &&
      tid == 0)
    atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
  if (q_len <= 0 || tok0 >= q_len) return;
  if (L < q_len || L > a.max_blocks_per_seq * bs) {
    if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
    return;
  }
  const int tok1 = min(tok0 + TPC, q_len);
  const int pos_base = a.causal ? L - q_len : -1;
  const int pos_first = a.causal ? pos_base + tok0 : L - 1;
  const int pos_last = a.causal ? pos_base + tok1 - 1 : L - 1;
  const int W = a.sliding_window;
  const int k_hi = pos_last + 1;
  const int k_lo = (W > 0 && pos_first + 1 > W) ? pos_first + 1 - W : 0;
  const int t_base = (k_lo / bs) * bs;
  const int ntiles = (k_hi - t_base + C::kKT - 1) / C::kKT;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw;
  const uint32_t s0 = smem_u32(smem);
  if (s0 & 1023u) {  // the swizzled tiles need 1024-byte alignment: refuse, do not guess
    if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SMEM);
    return;
  }
  const uint32_t q_s = s0 + C::kQOff;
  const uint32_t p_s = s0 + C::kPOff;
  const uint32_t ring_s = s0 + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::kStages;
  uint64_t* s_full = bars + 2 * C::kStages;   // [2]
  uint64_t* s_free = s_full + 2;              // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* fin_bar = o_done + 1;
  uint32_t* bad_copies = reinterpret_cast<uint32_t*>(smem + C::kBadOff);
  float* xmax = reinterpret_cast<float*>(smem + C::kXOff);
  float* lpart = reinterpret_cast<float*>(smem + C::kLOff);
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile int* abort_s = reinterpret_cast<volatile int*>(holder + 1);

  // ---- rows (softmax threads): row m = 32 (warp % 4) + lane, token m / G,
  // head m % G; the thread takes key columns [32 hf, 32 hf + 32) of the row
  // and head_dim columns [hf D / 2, (hf + 1) D / 2) of its output ----
  int rpos = -1, rlo = 0;
  bool rvalid = false;
  const uint16_t* qrow = nullptr;
  uint16_t* orow = nullptr;
  const int m = (warp & 3) * 32 + lane;
  const int hf = warp >> 2;
  if (warp < kSoftWarps) {
    const int t = tok0 + m / G;
    rvalid = (m / G) < TPC && t < tok1;
    const int tt = rvalid ? t : tok0;
    const int qh = g * G + m % G;
    rpos = rvalid ? (a.causal ? pos_base + tt : L - 1) : -1;
    rlo = (W > 0 && rpos + 1 > W) ? rpos + 1 - W : 0;
    qrow = a.q + static_cast<int64_t>(q0 + tt) * a.q_stride + static_cast<int64_t>(qh) * D;
    orow = a.out + static_cast<int64_t>(q0 + tt) * a.out_stride + static_cast<int64_t>(qh) * D;
    // this thread's half of the Q row into the K-major, 128-byte swizzled A
    // tile (zeros for padding rows)
#pragma unroll
    for (int pc = 0; pc < C::kDCH * 4; ++pc) {
      const int piece = hf * C::kDCH * 4 + pc;  // 16-byte piece of the row
      const int ch = piece / 8, q16 = piece % 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (rvalid) v = *reinterpret_cast<const uint4*>(qrow + ch * 64 + q16 * 8);
      sts128(q_s + ch * (kRowsU * 128) + swz128(m * 128 + q16 * 16), v.x, v.y, v.z, v.w);
    }
    fence_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t count = 1;
      const uint64_t* bb = bars + i;
      if (bb == &s_free[0] || bb == &s_free[1] || bb == p_full) count = kSoftWarps;
      mbar_init(smem_u32(bars + i), count);
    }
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(holder)),
                 "n"(tmem_cols<D>())
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  const uint32_t o_tmem = tmem + 128;
  bool failed = false;

  if (warp == kProdWarp) {
    // =========================== producer =================================
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    }
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
    const int pool_rows = static_cast<int>(a.num_blocks * bs);  // first row past the pool
    int cached_base = -(1 << 30);
    int my_entry = -1;
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % C::kStages;
      if (i >= C::kStages &&
          !warp_wait(smem_u32(&kv_empty[st]), ((i / C::kStages) - 1) & 1, abort_s)) {
        failed = true;
        break;
      }
      const int t0 = t_base + i * C::kKT;
      uint32_t bad = 0;
      int zrow[C::kNCopy];
#pragma unroll
      for (int j = 0; j < C::kNCopy; ++j) {
        const int tt = t0 + j * C::kBR;
        zrow[j] = pool_rows;  // a box past the pool: zero fill
        if (tt < k_hi) {
          const int pidx = tt / bs;
          if (pidx - cached_base >= 32 || pidx < cached_base) {  // warp-uniform refill
            cached_base = pidx;
            const int e = cached_base + lane;
            my_entry = (e < a.max_blocks_per_seq) ? bt[e] : -1;
          }
          const int pg = __shfl_sync(0xFFFFFFFFu, my_entry, pidx - cached_base);
          if (pg >= 0 && pg < a.num_blocks) zrow[j] = pg * bs + tt % bs;
          else bad |= 1u << j;
        }
      }
      const uint32_t fb = smem_u32(&kv_full[st]);
      if (lane == 0) {
        if (bad) atomicOr(a.flags, PD_DEV_BAD_PAGE);
        bad_copies[st] = bad;
        mbar_arrive_expect_tx(fb, 2u * C::kNCopy * C::kCopyBytes);
      }
      __syncwarp();
      if (lane < C::kNCopy) {
        const int j = lane;
        int z = pool_rows;
#pragma unroll
        for (int jj = 0; jj < C::kNCopy; ++jj)
          if (jj == j) z = zrow[jj];
        const uint32_t kst = ring_s + st * C::kStageBytes;
        const uint32_t vst = kst + C::kCacheStageBytes;
#pragma unroll
        for (int ch = 0; ch < C::kDCH; ++ch) {
          const uint32_t off = ch * (C::kKT * 128) + j * (C::kBR * 128);
          tma_load_3d(kst + off, &tm_k, ch * 64, g, z, fb);
          tma_load_3d(vst + off, &tm_v, ch * 64, g, z, fb);
        }
      }
      __syncwarp();
      issued = i + 1;
    }
    if (failed) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      *abort_s = 1;
      // let the copies already issued land before the block can exit
      for (int t = max(0, issued - C::kStages); t < issued; ++t)
        (void)mbar_wait(smem_u32(&kv_full[t % C::kStages]), (t / C::kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
    // =========================== MMA issuer ===============================
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc(kRowsU, C::kKT, 0);
      constexpr uint32_t idO = umma_idesc(kRowsU, D, 1);
      auto issue_s = [&](int j) -> bool {
        const int st = j % C::kStages;
        const int sb = j & 1;
        if (!mbar_wait(smem_u32(&kv_full[st]), (j / C::kStages) & 1)) return false;
        if (j >= 2 && !mbar_wait(smem_u32(&s_free[sb]), ((j - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kst = ring_s + st * C::kStageBytes;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          const uint32_t off = (ks >> 2) * (C::kKT * 128) + (ks & 3) * 32;
          const uint32_t qoff = (ks >> 2) * (kRowsU * 128) + (ks & 3) * 32;
          umma_f16(tmem + sb * 64, umma_desc(q_s + qoff, 16, 1024),
                   umma_desc(kst + off, 16, 1024), idS, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&s_full[sb]));
        return true;
      };
      bool ok = ntiles > 0 ? issue_s(0) : true;
      for (int j = 0; j < ntiles && ok; ++j) {
        if (j + 1 < ntiles && !(ok = issue_s(j + 1))) break;
        if (!(ok = mbar_wait(smem_u32(p_full), j & 1))) break;
        tc_fence_after();
        const uint32_t vst = ring_s + (j % C::kStages) * C::kStageBytes + C::kCacheStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_f16(o_tmem, umma_desc(p_s + kk * 32, 16, 1024),
                   umma_desc(vst + kk * 2048, 8192, 1024), idO, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(smem_u32(o_done));
        umma_commit(smem_u32(&kv_empty[j % C::kStages]));
      }
      if (!ok) {
        atomicOr(a.flags, PD_DEV_TIMEOUT);
        *abort_s = 1;
      }
      // every MMA issued so far has completed before TMEM is freed
      umma_commit(smem_u32(fin_bar));
      (void)mbar_wait(smem_u32(fin_bar), 0);
    }
    __syncwarp();
  } else {
    // =========================== softmax warps =============================
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    constexpr int kDH = D / 2;  // head_dim columns of O this thread rescales and writes
    float m_run = -INFINITY, l_part = 0.0f;
    // Every softmax warp reaches the row-max exchange (named barrier 1) once
    // per tile, even after a wait of its own gave up: it then skips every
    // further wait and all the work, so the barrier counts always match.
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % C::kStages;
      const int sb = j & 1;
      const int t0 = t_base + j * C::kKT;
      if (!failed && (!warp_wait(smem_u32(&kv_full[st]), (j / C::kStages) & 1, abort_s) ||
                      !warp_wait(smem_u32(&s_full[sb]), (j >> 1) & 1, abort_s)))
        failed = true;
      if (failed) {
        asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");
        continue;
      }
      tc_fence_after();
      const uint32_t bad = bad_copies[st];
      float s[32];  // keys t0 + 32 hf + k
      {
        uint32_t v[2][16];
        tmem_ld16(tmem + lane_base + sb * 64 + hf * 32, v[0]);
        tmem_ld16(tmem + lane_base + sb * 64 + hf * 32 + 16, v[1]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          s[k] = __uint_as_float(v[0][k]);
          s[16 + k] = __uint_as_float(v[1][k]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));

      // ---- mask and scale; the row max from both halves ----
      // bit k of `valid`: key t0 + 32 hf + k is in [rlo, rpos] and its page is
      // in the pool (built once per tile, so the element loop has no branches)
      const int k0 = t0 + hf * 32;
      const int klo = max(rlo - k0, 0), khi = min(rpos + 1 - k0, 32);  // [klo, khi)
      uint32_t valid = 0u;
      if (khi > klo)
        valid = (khi - klo == 32 ? 0xFFFFFFFFu : ((1u << (khi - klo)) - 1u)) << klo;
      if (bad) {
#pragma unroll
        for (int c = 0; c < 32 / C::kBR + (C::kBR > 32 ? 1 : 0); ++c) {
          const int copy = (hf * 32 + c * C::kBR) / C::kBR;
          if ((bad >> copy) & 1u)
            valid &= ~((C::kBR >= 32 ? 0xFFFFFFFFu : ((1u << C::kBR) - 1u)) << (c * C::kBR));
        }
      }
      float mxp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (valid == 0xFFFFFFFFu) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] *= sl2;
          mxp[k & 3] = fmaxf(mxp[k & 3], s[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] = ((valid >> k) & 1u) ? s[k] * sl2 : -INFINITY;
          mxp[k & 3] = fmaxf(mxp[k & 3], s[k]);
        }
      }
      const float mh = fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3]));
      xmax[(sb * 2 + hf) * kRowsU + m] = mh;
      asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");
      const float mx = fmaxf(mh, xmax[(sb * 2 + (hf ^ 1)) * kRowsU + m]);
      // the reference max moves only past the threshold (or from -inf)
      const float mn = (mx > m_run + kRescaleLog2) ? mx : m_run;
      const float alpha = (mn == m_run) ? 1.0f : ex2(m_run - mn);
      float lsp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (mn == -INFINITY) {  // nothing seen yet by this row: P = 0
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = 0.0f;
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] = ex2(s[k] - mn);
          lsp[k & 3] += s[k];
        }
      }
      l_part = l_part * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
      m_run = mn;

      // ---- V rows no row of the CTA may read: zero them (stale bytes) ----
      const bool ragged = t0 < k_lo || t0 + C::kKT > k_hi || bad != 0u;
      if (ragged) {
        const uint32_t vst = ring_s + st * C::kStageBytes + C::kCacheStageBytes;
        constexpr int kPieces = C::kKT * C::kDCH * 8;  // 16-byte pieces in the V tile
        const int t = hf * kRowsU + m;                 // 0 .. 255
        for (int pc = t; pc < kPieces; pc += kSoftWarps * 32) {
          const int ch = pc / (C::kKT * 8);
          const int key = (pc / 8) % C::kKT;
          const int kabs = t0 + key;
          const bool keep = kabs >= k_lo && kabs < k_hi && !((bad >> (key / C::kBR)) & 1u);
          if (!keep)
            sts128(vst + ch * (C::kKT * 128) + swz128(key * 128 + (pc % 8) * 16), 0u, 0u, 0u,
                   0u);
        }
      }

      // ---- P_j may replace P_{j-1} and O may be rescaled once PV_{j-1} is done ----
      if (j > 0) {
        if (!warp_wait(smem_u32(o_done), (j - 1) & 1, abort_s)) {
          failed = true;
          continue;  // the next tiles still reach the exchange barrier
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll
          for (int h = 0; h < kDH / 32; ++h) {  // 32 of this thread's columns at a time
            uint32_t v[2][16];
            const uint32_t col = o_tmem + lane_base + hf * kDH + h * 32;
            tmem_ld16(col, v[0]);
            tmem_ld16(col + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int cg = 0; cg < 2; ++cg) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                v[cg][k] = __float_as_uint(__uint_as_float(v[cg][k]) * alpha);
              tmem_st16(col + cg * 16, v[cg]);
            }
          }
          tmem_wait_st();
        }
      }
      // P row m, keys [32 hf, 32 hf + 32): four swizzled 16-byte pieces
#pragma unroll
      for (int q = 0; q < 4; ++q)
        sts128(p_s + swz128(m * 128 + (hf * 4 + q) * 16),
               pack_bf16x2(s[q * 8 + 0], s[q * 8 + 1]), pack_bf16x2(s[q * 8 + 2], s[q * 8 + 3]),
               pack_bf16x2(s[q * 8 + 4], s[q * 8 + 5]), pack_bf16x2(s[q * 8 + 6], s[q * 8 + 7]));
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    // ---- epilogue: out = O / l, l from both halves of the row ----
    lpart[hf * kRowsU + m] = l_part;
    asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");
    const float l_row = l_part + lpart[(hf ^ 1) * kRowsU + m];
    if (!failed && ntiles > 0) {
      if (!warp_wait(smem_u32(o_done), (ntiles - 1) & 1, abort_s)) {
        failed = true;
      } else {
        tc_fence_after();
        const float inv = 1.0f / fmaxf(l_row, 1e-20f);
#pragma unroll
        for (int cg = 0; cg < kDH / 16; ++cg) {
          uint32_t v[16];
          tmem_ld16(o_tmem + lane_base + hf * kDH + cg * 16, v);
          tmem_wait_ld();
          if (rvalid) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * inv,
                                 __uint_as_float(v[2 * k + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(orow + hf * kDH + cg * 16);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
    if (failed) {
      if (lane == 0) atomicOr(a.flags, PD_DEV_TIMEOUT);
      *abort_s = 1;
    }
  }

  // ---- free the TMEM columns once every warp is done with them ----
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(tmem_cols<D>())
                 : "memory");
  }
}

template <int D, int BS>
cudaError_t launch_umma_cfg(const PrefillArgs& a, const void* kc, const void* vc, int max_q_len,
                            cudaStream_t st) {
  using C = UCfg<D, BS>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  const int64_t rows = a.num_blocks * a.block_size;
  if (!encode_cache_map(&tk, kc, PD_KV_BF16, D, a.num_kv_heads, rows, 64, C::kBR, true) ||
      !encode_cache_map(&tv, vc, PD_KV_BF16, D, a.num_kv_heads, rows, 64, C::kBR, true))
    return cudaErrorInvalidValue;
  auto kern = prefill_umma_kernel<D, BS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int tiles = (max_q_len + a.tokens_per_cta - 1) / a.tokens_per_cta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(kUmmaThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

}  // namespace

cudaError_t launch_prefill_umma(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                                int head_dim, int max_q_len, cudaStream_t st) {
  if (a.num_seqs == 0 || max_q_len == 0) return cudaSuccess;
  const bool bs16 = a.block_size == 16;
  switch (head_dim) {  // head_dim 64 and 128 run on the two-tile kernel (prefill_pair.cu)
    case 256:
      return bs16 ? launch_umma_cfg<256, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_umma_cfg<256, 32>(a, k_cache, v_cache, max_q_len, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pd
