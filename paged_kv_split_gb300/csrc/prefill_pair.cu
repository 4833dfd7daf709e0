// Paged prefill on tcgen05 with two query tiles per CTA (head_dim 64 and 128,
// BF16 cache). Same semantics and interface as prefill_umma.cu's kernel
// (pegainfer issue 1008, `prefill_paged_launch`; AstrAI "csrc/tests" log:
// causal offset, stride addressing), which keeps head_dim 256. Design:
//
//  * One CTA per (pair of query tiles, kv head, sequence). Tile A holds the
//    first 128 (token, q head) rows of the pair, tile B the next 128 (128 / G
//    tokens each, all G heads of the GQA group). Both tiles read the same K/V
//    stages, so every stage loaded serves 256 rows, and while one tile's
//    softmax runs the tensor core works on the other tile's products.
//  * Warp 8 (producer) copies 64-key K and V tiles with 3-D TMA (128-byte
//    swizzle) over the union of the two tiles' key ranges, one block-table
//    lookup per page; copies it skips (pages outside the pool, rows past the
//    keys) are issued at a row past the pool and land as zeros.
//  * Warp 9 holds 512 TMEM columns: S of tile X in two buffers at X * 128 +
//    {0, 64}, O of tile X at 256 + X * 128. One thread issues, per key tile j,
//    S_X(j + 1) for both tiles ahead of time, then PV_A(j) and PV_B(j) once
//    the tiles' P are written, and releases the stage after both.
//  * Warps 0-3 run tile A's softmax, warps 4-7 tile B's: one thread per row
//    (TMEM lane = row), so a row's max, exponentials and sum stay in one
//    thread and no barrier joins the warps. Per tile a thread reads its 64
//    scores with tcgen05.ld, masks them with one 64-bit valid-key word
//    (causal position, window, pages outside the pool), takes P = 2^(s - m)
//    against a reference max m that moves only when the tile max passes it by
//    more than 2^8 (then O is rescaled in TMEM), and writes P as bf16 into
//    the tile's swizzled A-operand buffer. V rows no row of the CTA may read
//    are zeroed first (stale stage bytes never meet a zero weight).
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

constexpr float kRescaleLog2P = 8.0f;  // P <= 2^8 between rescales of O
constexpr int kPairSoftWarps = 8;      // warps 0-3: tile A, 4-7: tile B
constexpr int kPairProdWarp = 8;
constexpr int kPairMmaWarp = 9;
constexpr int kPairThreads = 10 * 32;
constexpr int kPairTmemCols = 512;
constexpr int kMaxRanked = 256;  // (sequence, pair) items a CTA ranks by cost

template <int D, int BS>
struct PairCfg {
  static constexpr int kKT = 64;                      // keys per stage (UMMA N of S)
  static constexpr int kBR = kKT < BS ? kKT : BS;     // rows per copy
  static constexpr int kNCopy = kKT / kBR;
  static constexpr int kDCH = D / 64;                 // 128-byte chunks per row
  static constexpr int kQBytes = kDCH * 128 * 128;    // one Q tile, chunk-major
  static constexpr int kPBytes = 128 * 128;           // one P tile: 128 rows x 64 keys
  static constexpr int kCacheStageBytes = kKT * 2 * D;
  static constexpr int kStageBytes = 2 * kCacheStageBytes;
  static constexpr int kStages = D == 128 ? 4 : 6;
  static constexpr int kQOff = 0;                     // Q_A, Q_B
  static constexpr int kPOff = 2 * kQBytes;           // P_A, P_B
  static constexpr int kRingOff = kPOff + 2 * kPBytes;
  static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
  // kv_full[S], kv_empty[S]; per tile: s_full[2], s_free[2], p_full, o_done; fin
  static constexpr int kTileBars = 6;
  static constexpr int kNumBars = 2 * kStages + 2 * kTileBars + 1;
  static constexpr int kBadOff = kBarOff + kNumBars * 8;
  static constexpr int kHolderOff = kBadOff + kStages * 4;
  static constexpr int kSmemBytes = kHolderOff + 16;
  static constexpr uint32_t kCopyBytes = kBR * 2 * D;
  static constexpr int kKS = D / 16;  // K steps of S
  static_assert(D == 64 || D == 128, "two query tiles need head_dim <= 128 (TMEM columns)");
  static_assert(kCacheStageBytes % 1024 == 0 && kQBytes % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
};

template <int D, int BS>
__global__ void __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  using C = PairCfg<D, BS>;
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int G = a.group;
  const int TPC = a.tokens_per_cta;  // tokens of one query tile: 128 / G
  const int bs = a.block_size;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw;
  const uint32_t s0 = smem_u32(smem);
  if (s0 & 1023u) {  // the swizzled tiles need 1024-byte alignment: refuse, do not guess
    if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SMEM);
    return;
  }

  // ---- which (sequence, pair of query tiles) and kv head this CTA takes ----
  // CTAs start in launch order (blockIdx.x fastest), one per SM at a time, so
  // the grid runs as a list schedule: CTA k takes the (k / Hkv)-th costliest
  // (sequence, pair) item, costs being the pair's key tiles plus two for its
  // start and end (longest first bounds the tail). Every CTA ranks all items
  // itself, from cu_q and seq_lens; above kMaxRanked items it takes them in
  // grid order instead, each sequence's last pair (the most keys) first.
  int g, b, pair;
  {
    const int PM = gridDim.x;  // pair slots per sequence
    const int n = PM * static_cast<int>(gridDim.z);
    if (n <= kMaxRanked) {
      const int k = blockIdx.x + PM * (blockIdx.y + gridDim.y * blockIdx.z);
      g = k % gridDim.y;
      const int r = k / gridDim.y;
      int* cost_s = reinterpret_cast<int*>(smem + C::kPOff);  // P buffers: free until then
      volatile int* pick_s = cost_s + kMaxRanked;
      for (int i = tid; i < n; i += kPairThreads) {
        const int bi = i / PM, t0 = (i % PM) * 2 * TPC;
        const int ql = a.cu_q[bi + 1] - a.cu_q[bi];
        const int Li = a.seq_lens[bi];
        int c = -1;  // no query rows: ranked last
        if (ql > 0 && t0 < ql) {
          c = 0;
          if (Li >= ql && Li <= a.max_blocks_per_seq * bs) {
            const int pf = a.causal ? Li - ql + t0 : Li - 1;
            const int pl = a.causal ? Li - ql + min(t0 + 2 * TPC, ql) - 1 : Li - 1;
            const int lo = (a.sliding_window > 0 && pf + 1 > a.sliding_window)
                               ? pf + 1 - a.sliding_window
                               : 0;
            c = (pl + 1 - (lo / bs) * bs + C::kKT - 1) / C::kKT + 2;
          }
        }
        cost_s[i] = c;
      }
      __syncthreads();
      for (int i = tid; i < n; i += kPairThreads) {
        const int ci = cost_s[i];
        int rank = 0;
        for (int j2 = 0; j2 < n; ++j2) {
          const int cj = cost_s[j2];
          rank += (cj > ci || (cj == ci && j2 < i)) ? 1 : 0;
        }
        if (rank == r) *pick_s = i;
      }
      __syncthreads();
      const int item = *pick_s;
      b = item / PM;
      pair = item % PM;
    } else {
      g = blockIdx.y;
      b = blockIdx.z;
      pair = PM - 1 - blockIdx.x;
    }
  }

  // ---- the pair's query tokens and the keys each tile may see ----
  const int q0 = a.cu_q[b];
  const int q_len = a.cu_q[b + 1] - q0;
  const int L = a.seq_lens[b];
  const int tok0 = pair * 2 * TPC;
  if (pair == static_cast<int>(gridDim.x) - 1 && q_len > static_cast<int>(gridDim.x) * 2 * TPC &&
      tid == 0)
    atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
  if (q_len <= 0 || tok0 >= q_len) return;
  if (L < q_len || L > a.max_blocks_per_seq * bs) {
    if (tid == 0) atomicOr(a.flags, PD_DEV_BAD_SEQ_LEN);
    return;
  }
  const int W = a.sliding_window;
  const int pos_base = a.causal ? L - q_len : -1;
  auto pos_of = [&](int t) { return a.causal ? pos_base + t : L - 1; };
  // tile x: tokens [tx0(x), tx1(x)); key range [klo, khi); key tiles
  // [j0(x), j1(x)) of the pair's tile line (empty for a tile past q_len).
  // Scalars per tile, not arrays: a runtime tile index must not put them in
  // local memory.
  const int txA0 = tok0, txA1 = min(tok0 + TPC, q_len);
  const int txB0 = tok0 + TPC, txB1 = min(tok0 + 2 * TPC, q_len);
  const bool hasB = txB1 > txB0;
  auto key_lo = [&](int t) {
    const int p = pos_of(t);
    return (W > 0 && p + 1 > W) ? p + 1 - W : 0;
  };
  const int kloA = key_lo(txA0), khiA = pos_of(txA1 - 1) + 1;
  const int kloB = hasB ? key_lo(txB0) : 0, khiB = hasB ? pos_of(txB1 - 1) + 1 : 0;
  const int k_lo = kloA;                   // union of both tiles' keys
  const int k_hi = hasB ? khiB : khiA;
  const int t_base = (k_lo / bs) * bs;
  const int ntiles = (k_hi - t_base + C::kKT - 1) / C::kKT;
  const int jA0 = (kloA - t_base) / C::kKT, jA1 = (khiA - t_base + C::kKT - 1) / C::kKT;
  const int jB0 = hasB ? (kloB - t_base) / C::kKT : 0;
  const int jB1 = hasB ? (khiB - t_base + C::kKT - 1) / C::kKT : 0;
  auto j0 = [&](int x) { return x ? jB0 : jA0; };
  auto j1 = [&](int x) { return x ? jB1 : jA1; };

  const uint32_t ring_s = s0 + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::kStages;
  uint64_t* tile_bars = bars + 2 * C::kStages;  // tile X: tile_bars + X * kTileBars
  uint64_t* fin_bar = tile_bars + 2 * C::kTileBars;
  auto s_full = [&](int X, int i) { return tile_bars + X * C::kTileBars + i; };
  auto s_free = [&](int X, int i) { return tile_bars + X * C::kTileBars + 2 + i; };
  auto p_full = [&](int X) { return tile_bars + X * C::kTileBars + 4; };
  auto o_done = [&](int X) { return tile_bars + X * C::kTileBars + 5; };
  uint32_t* bad_copies = reinterpret_cast<uint32_t*>(smem + C::kBadOff);
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile int* abort_s = reinterpret_cast<volatile int*>(holder + 1);

  // ---- softmax threads: tile X = warp / 4, row m = 32 (warp % 4) + lane,
  // token m / G, head m % G ----
  const int X = warp >> 2;
  const int m = (warp & 3) * 32 + lane;
  int rpos = -1, rlo = 0;
  bool rvalid = false;
  uint16_t* orow = nullptr;
  if (warp < kPairSoftWarps) {
    const int t = (X ? txB0 : txA0) + m / G;
    rvalid = (m / G) < TPC && t < (X ? txB1 : txA1);
    const int tt = rvalid ? t : tok0;
    const int qh = g * G + m % G;
    rpos = rvalid ? pos_of(tt) : -1;
    rlo = (W > 0 && rpos + 1 > W) ? rpos + 1 - W : 0;
    const uint16_t* qrow =
        a.q + static_cast<int64_t>(q0 + tt) * a.q_stride + static_cast<int64_t>(qh) * D;
    orow = a.out + static_cast<int64_t>(q0 + tt) * a.out_stride + static_cast<int64_t>(qh) * D;
    // the Q row into tile X's K-major, 128-byte swizzled A tile (zeros for
    // padding rows)
    const uint32_t q_s = s0 + C::kQOff + X * C::kQBytes;
#pragma unroll
    for (int piece = 0; piece < C::kDCH * 8; ++piece) {  // 16-byte pieces of the row
      const int ch = piece / 8, q16 = piece % 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (rvalid) v = *reinterpret_cast<const uint4*>(qrow + ch * 64 + q16 * 8);
      sts128(q_s + ch * (128 * 128) + swz128(m * 128 + q16 * 16), v.x, v.y, v.z, v.w);
    }
    fence_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t count = 1;
      const uint64_t* bb = bars + i;
      for (int x = 0; x < 2; ++x)
        if (bb == s_free(x, 0) || bb == s_free(x, 1) || bb == p_full(x)) count = 4;
      mbar_init(smem_u32(bars + i), count);
    }
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kPairMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(holder)),
                 "n"(kPairTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  bool failed = false;

  if (warp == kPairProdWarp) {
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
  } else if (warp == kPairMmaWarp) {
    // =========================== MMA issuer ===============================
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc(128, C::kKT, 0);
      constexpr uint32_t idO = umma_idesc(128, D, 1);
      // Descriptors are built once: a descriptor's start-address field is the
      // byte address / 16, so an offset inside a tile is a constant added to
      // its low word (tiles stay below 256 KB of shared memory). One thread
      // issues every MMA: per instruction an add and the MMA itself.
      const uint64_t dqA = umma_desc(s0 + C::kQOff, 16, 1024);
      const uint64_t dqB = umma_desc(s0 + C::kQOff + C::kQBytes, 16, 1024);
      const uint64_t dpA = umma_desc(s0 + C::kPOff, 16, 1024);
      const uint64_t dpB = umma_desc(s0 + C::kPOff + C::kPBytes, 16, 1024);
      const uint64_t dk0 = umma_desc(ring_s, 16, 1024);
      const uint64_t dv0 = umma_desc(ring_s + C::kCacheStageBytes, 8192, 1024);
      // S_x(j) = Q_x K_j^T into buffer (j - j0(x)) & 1 of tile x
      auto issue_s = [&](int x, int j) -> bool {
        const int jl = j - j0(x);
        const int st = j % C::kStages;
        if (!mbar_wait(smem_u32(&kv_full[st]), (j / C::kStages) & 1)) return false;
        if (jl >= 2 && !mbar_wait(smem_u32(s_free(x, jl & 1)), ((jl - 2) >> 1) & 1))
          return false;
        tc_fence_after();
        const uint64_t a0 = x ? dqB : dqA;
        const uint64_t b0 = dk0 + static_cast<uint64_t>((st * C::kStageBytes) >> 4);
        const uint32_t d = tmem + x * 128 + (jl & 1) * 64;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          constexpr int kQChunk = 128 * 128, kKChunk = C::kKT * 128;
          const uint32_t qoff = ((ks >> 2) * kQChunk + (ks & 3) * 32) >> 4;
          const uint32_t koff = ((ks >> 2) * kKChunk + (ks & 3) * 32) >> 4;
          umma_f16(d, a0 + qoff, b0 + koff, idS, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(s_full(x, jl & 1)));
        return true;
      };
      int nsA = jA0, nsB = jB0;  // next S tile to issue per query tile
      bool ok = true;
      for (int j = 0; j < ntiles && ok; ++j) {
        // S of the next key tile for both query tiles, ahead of this tile's PV
        while (ok && nsA < jA1 && nsA <= j + 1) ok = issue_s(0, nsA++);
        while (ok && nsB < jB1 && nsB <= j + 1) ok = issue_s(1, nsB++);
        if (!ok) break;
        const uint64_t bv = dv0 + static_cast<uint64_t>(((j % C::kStages) * C::kStageBytes) >> 4);
        for (int x = 0; x < 2; ++x) {
          if (j < j0(x) || j >= j1(x)) continue;
          const int jl = j - j0(x);
          if (!(ok = mbar_wait(smem_u32(p_full(x)), jl & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem + 256 + x * 128, (x ? dpB : dpA) + ((kk * 32) >> 4), bv + ((kk * 2048) >> 4),
                     idO, (jl > 0 || kk > 0) ? 1u : 0u);
          umma_commit(smem_u32(o_done(x)));
        }
        if (!ok) break;
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
    const uint32_t s_tm = tmem + lane_base + X * 128;
    const uint32_t o_tm = tmem + lane_base + 256 + X * 128;
    const uint32_t p_s = s0 + C::kPOff + X * C::kPBytes;
    const float sl2 = a.scale_log2;
    const int jX0 = j0(X);
    const int nX = j1(X) - jX0;
    float m_run = -INFINITY, l_run = 0.0f;
    for (int jl = 0; jl < nX && !failed; ++jl) {
      const int j = jX0 + jl;
      const int st = j % C::kStages;
      const int sb = jl & 1;
      const int t0 = t_base + j * C::kKT;
      if (!warp_wait(smem_u32(&kv_full[st]), (j / C::kStages) & 1, abort_s) ||
          !warp_wait(smem_u32(s_full(X, sb)), (jl >> 1) & 1, abort_s)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t bad = bad_copies[st];
      // ---- bit k of `valid`: key t0 + k is in [rlo, rpos] and its page in
      // the pool ----
      const int klo_r = max(rlo - t0, 0), khi_r = min(rpos + 1 - t0, 64);  // [klo_r, khi_r)
      uint64_t valid = 0ull;
      if (khi_r > klo_r)
        valid = (khi_r - klo_r == 64 ? ~0ull : ((1ull << (khi_r - klo_r)) - 1ull)) << klo_r;
      if (bad) {
#pragma unroll
        for (int c = 0; c < C::kNCopy; ++c)
          if ((bad >> c) & 1u)
            valid &= ~((C::kBR >= 64 ? ~0ull : ((1ull << C::kBR) - 1ull)) << (c * C::kBR));
      }
      // A full tile of a row that has seen keys takes P = 2^(s scale log2e -
      // m_run) against the current reference right away, the first 32 scores
      // while the last 32 are still on their way from TMEM. Only if the tile
      // passes the reference by more than the threshold does the warp read
      // the scores again and take P against the new reference (the same
      // rule as taking the tile max first). Other tiles (the row's first,
      // masked ones) take the max first.
      const bool fast = valid == ~0ull && m_run != -INFINITY;
      const uint32_t sbase = s_tm + sb * 64;
      float p[64];
      float lsp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      float mn = m_run, alpha = 1.0f;
      {
        uint32_t v[4][16];
        tmem_ld16(sbase, v[0]);
        tmem_ld16(sbase + 16, v[1]);
        tmem_wait_ld();
        tmem_ld16(sbase + 32, v[2]);
        tmem_ld16(sbase + 48, v[3]);
        float mxp[2] = {-INFINITY, -INFINITY};
        const float nref = -m_run;
        if (fast) {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float x = fmaf(__uint_as_float(v[k >> 4][k & 15]), sl2, nref);
            mxp[k & 1] = fmaxf(mxp[k & 1], x);
            p[k] = ex2(x);
            lsp[k & 3] += p[k];
          }
        }
        tmem_wait_ld();
        if (fast) {
#pragma unroll
          for (int k = 32; k < 64; ++k) {
            const float x = fmaf(__uint_as_float(v[k >> 4][k & 15]), sl2, nref);
            mxp[k & 1] = fmaxf(mxp[k & 1], x);
            p[k] = ex2(x);
            lsp[k & 3] += p[k];
          }
          const float mx = fmaxf(mxp[0], mxp[1]);  // tile max above the reference
          if (mx > kRescaleLog2P) {
            mn = m_run + mx;
            alpha = ex2(-mx);
          }
        } else {
          float mxq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            const float x = ((valid >> k) & 1ull) ? __uint_as_float(v[k >> 4][k & 15]) * sl2
                                                  : -INFINITY;
            p[k] = x;
            mxq[k & 3] = fmaxf(mxq[k & 3], x);
          }
          const float mx = fmaxf(fmaxf(mxq[0], mxq[1]), fmaxf(mxq[2], mxq[3]));
          // the reference max moves only past the threshold (or from -inf)
          mn = (mx > m_run + kRescaleLog2P) ? mx : m_run;
          alpha = (mn == m_run) ? 1.0f : ex2(m_run - mn);
          if (mn == -INFINITY) {  // nothing seen yet by this row: P = 0
#pragma unroll
            for (int k = 0; k < 64; ++k) p[k] = 0.0f;
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              p[k] = ex2(p[k] - mn);
              lsp[k & 3] += p[k];
            }
          }
        }
        // a fast row whose reference moved: the scores again, P against it
        const bool redo = fast && mn != m_run;
        if (__any_sync(0xFFFFFFFFu, redo)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(sbase + c * 16, v[c]);
          tmem_wait_ld();
          if (redo) {
            const float nr = -mn;
#pragma unroll
            for (int q = 0; q < 4; ++q) lsp[q] = 0.0f;
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              p[k] = ex2(fmaf(__uint_as_float(v[k >> 4][k & 15]), sl2, nr));
              lsp[k & 3] += p[k];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(s_free(X, sb)));
      l_run = l_run * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
      m_run = mn;

      // ---- V rows no row of the CTA may read: zeroed (stale bytes) by the
      // first query tile that reads the stage, before its P is released ----
      const bool zeroer = (X == 0) || j < jA0 || j >= jA1;
      const bool ragged = t0 < k_lo || t0 + C::kKT > k_hi || bad != 0u;
      if (zeroer && ragged) {
        const uint32_t vst = ring_s + st * C::kStageBytes + C::kCacheStageBytes;
        constexpr int kPieces = C::kKT * C::kDCH * 8;  // 16-byte pieces in the V tile
        for (int pc = m; pc < kPieces; pc += 128) {
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
      if (jl > 0) {
        if (!warp_wait(smem_u32(o_done(X)), (jl - 1) & 1, abort_s)) {
          failed = true;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll
          for (int h = 0; h < D / 32; ++h) {  // 32 columns of the row at a time
            uint32_t v[2][16];
            tmem_ld16(o_tm + h * 32, v[0]);
            tmem_ld16(o_tm + h * 32 + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int cg = 0; cg < 2; ++cg) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                v[cg][k] = __float_as_uint(__uint_as_float(v[cg][k]) * alpha);
              tmem_st16(o_tm + h * 32 + cg * 16, v[cg]);
            }
          }
          tmem_wait_st();
        }
      }
      // P row m, keys 0..63: eight swizzled 16-byte pieces
#pragma unroll
      for (int q = 0; q < 8; ++q)
        sts128(p_s + swz128(m * 128 + q * 16), pack_bf16x2(p[q * 8 + 0], p[q * 8 + 1]),
               pack_bf16x2(p[q * 8 + 2], p[q * 8 + 3]), pack_bf16x2(p[q * 8 + 4], p[q * 8 + 5]),
               pack_bf16x2(p[q * 8 + 6], p[q * 8 + 7]));
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full(X)));
    }
    // ---- epilogue: out = O / l ----
    if (!failed && nX > 0) {
      if (!warp_wait(smem_u32(o_done(X)), (nX - 1) & 1, abort_s)) {
        failed = true;
      } else {
        tc_fence_after();
        const float inv = 1.0f / fmaxf(l_run, 1e-20f);
#pragma unroll
        for (int cg = 0; cg < D / 16; ++cg) {
          uint32_t v[16];
          tmem_ld16(o_tm + cg * 16, v);
          tmem_wait_ld();
          if (rvalid) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * inv,
                                 __uint_as_float(v[2 * k + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(orow + cg * 16);
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
  if (warp == kPairMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(kPairTmemCols)
                 : "memory");
  }
}

template <int D, int BS>
cudaError_t launch_pair_cfg(const PrefillArgs& a, const void* kc, const void* vc, int max_q_len,
                            cudaStream_t st) {
  using C = PairCfg<D, BS>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  const int64_t rows = a.num_blocks * a.block_size;
  if (!encode_cache_map(&tk, kc, PD_KV_BF16, D, a.num_kv_heads, rows, 64, C::kBR, true) ||
      !encode_cache_map(&tv, vc, PD_KV_BF16, D, a.num_kv_heads, rows, 64, C::kBR, true))
    return cudaErrorInvalidValue;
  auto kern = prefill_pair_kernel<D, BS>;
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
  const int pairs = (max_q_len + 2 * a.tokens_per_cta - 1) / (2 * a.tokens_per_cta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs, a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(kPairThreads);
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

cudaError_t launch_prefill_pair(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                                int head_dim, int max_q_len, cudaStream_t st) {
  if (a.num_seqs == 0 || max_q_len == 0) return cudaSuccess;
  const bool bs16 = a.block_size == 16;
  switch (head_dim) {
    case 64:
      return bs16 ? launch_pair_cfg<64, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_pair_cfg<64, 32>(a, k_cache, v_cache, max_q_len, st);
    case 128:
      return bs16 ? launch_pair_cfg<128, 16>(a, k_cache, v_cache, max_q_len, st)
                  : launch_pair_cfg<128, 32>(a, k_cache, v_cache, max_q_len, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pd
