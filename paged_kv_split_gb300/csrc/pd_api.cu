// The C ABI of libpd.so (declared in include/pd.h): argument validation, the
// split planner and dispatch to the kernels. Nothing here allocates device
// memory or synchronises, except pd_device_status (a debugging read).
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <mutex>
#include <vector>

#include "pd_common.cuh"

namespace pd {
namespace {

// Device status word (pd_device_flag bits); kernels get its device address.
__device__ int g_device_flags;

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 1024;

struct DeviceInfo {
  std::once_flag once;
  int num_sms = 0;
  int* flags = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceInfo g_devices[kMaxDevices];

// Limit of the decode kernels' consumer-side waits (ns). Only a test changes
// it (pd_test_set_consumer_wait_ns), to make those waits run out on purpose.
constexpr uint32_t kDefaultConsumerWaitNs = 2000000000u;
std::atomic<uint32_t> g_consumer_wait_ns{kDefaultConsumerWaitNs};

// SM count and status-word address of the current device (looked up once).
cudaError_t current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceInfo& d = g_devices[dev];
  std::call_once(d.once, [&d, dev]() {
    d.err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.err == cudaSuccess)
      d.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.flags), g_device_flags);
  });
  *out = &d;
  return d.err;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dev_ptr_ok(const void* p) { return p != nullptr && aligned16(p); }
bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }
bool block_size_ok(int bs) { return bs == 16 || bs == 32; }
bool dtype_ok(int t) { return t == PD_KV_BF16 || t == PD_KV_FP8_E4M3 || t == PD_KV_NVFP4; }
bool scale_ok(float s) { return isfinite(s) && s > 0.0f; }

struct DecodeShape {
  int B, Hq, Hkv, D, bs, mbs, S, W, kv_dtype;
  int64_t nb;
};

// Shape and scale checks of every decode call (no pointer, split count or
// workspace involved), in the order the status codes are reported.
int check_decode_shape(const DecodeShape& s, float k_scale, float v_scale) {
  if (s.B < 0 || s.B > 65535) return PD_ERR_INVALID_ARG;
  if (s.Hkv <= 0 || s.Hq <= 0 || s.Hq % s.Hkv != 0) return PD_ERR_INVALID_ARG;
  if (s.Hq / s.Hkv > kMaxGroup) return PD_ERR_UNSUPPORTED;
  if (!head_dim_ok(s.D) || !block_size_ok(s.bs)) return PD_ERR_UNSUPPORTED;
  if (!dtype_ok(s.kv_dtype)) return PD_ERR_UNSUPPORTED;
  if (s.mbs <= 0 || s.nb <= 0 || s.W < 0) return PD_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s.mbs) * s.bs > (int64_t{1} << 30)) return PD_ERR_INVALID_ARG;
  if (s.nb * s.bs > INT32_MAX) return PD_ERR_INVALID_ARG;  // pool rows are int32 coordinates
  if (s.kv_dtype == PD_KV_FP8_E4M3 && !(scale_ok(k_scale) && scale_ok(v_scale)))
    return PD_ERR_INVALID_ARG;
  return PD_OK;
}

// Shared checks of pd_decode / pd_decode_partial (S already resolved).
int check_decode(const DecodeShape& s, const void* q, const void* kc, const void* vc,
                 const int32_t* bt, const int32_t* lens, float k_scale, float v_scale,
                 const void* ws, size_t ws_bytes) {
  const int rc = check_decode_shape(s, k_scale, v_scale);
  if (rc != PD_OK) return rc;
  if (s.S < 1 || s.S > kMaxSplits) return PD_ERR_INVALID_ARG;
  if (s.B == 0) return PD_OK;
  if (!dev_ptr_ok(q) || !dev_ptr_ok(kc) || !dev_ptr_ok(vc) || !dev_ptr_ok(bt) ||
      !dev_ptr_ok(lens) || !dev_ptr_ok(ws))
    return PD_ERR_INVALID_ARG;
  if (ws_bytes < ws_total_bytes(s.B, s.Hq, s.D, s.S)) return PD_ERR_WORKSPACE_TOO_SMALL;
  return PD_OK;
}

DecodeArgs make_decode_args(const DecodeShape& s, const void* q, const void* kc, const void* vc,
                            const int32_t* bt, const int32_t* lens, float scale, float k_scale,
                            float v_scale, void* ws, int* flags) {
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.q_stride = static_cast<int64_t>(s.Hq) * s.D;
  a.k_cache = static_cast<const uint8_t*>(kc);
  a.v_cache = static_cast<const uint8_t*>(vc);
  a.block_tables = bt;
  a.seq_lens = lens;
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + ws_o_bytes(s.B, s.Hq, s.D, s.S));
  a.flags = flags;
  a.out = nullptr;
  a.out_stride = static_cast<int64_t>(s.Hq) * s.D;
  a.direct = 0;
  a.num_blocks = s.nb;
  a.page_bytes = page_bytes_of(s.kv_dtype, s.bs, s.Hkv, s.D);
  a.data_bytes = nvfp4_data_bytes(s.bs, s.Hkv, s.D);
  a.num_seqs = s.B;
  a.num_q_heads = s.Hq;
  a.num_kv_heads = s.Hkv;
  a.group = s.Hq / s.Hkv;
  a.block_size = s.bs;
  a.max_blocks_per_seq = s.mbs;
  a.num_splits = s.S;
  a.chunk = chunk_pages(page_span_max(s.mbs, s.bs, s.W), s.S);
  a.sliding_window = s.W;
  a.plan_cta = nullptr;
  a.plan_pieces = nullptr;
  a.plan_num_ctas = 0;
  a.plan_num_pieces = 0;
  a.scale_log2 = scale * kLog2e;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.consumer_wait_ns = g_consumer_wait_ns.load(std::memory_order_relaxed);
  return a;
}

CombineArgs make_combine_args(int B, int Hq, int D, int bs, int mbs, int S, int W, const void* ws,
                              const int32_t* lens, void* out) {
  CombineArgs c;
  c.ws_o = static_cast<const float*>(ws);
  c.ws_ml = reinterpret_cast<const float2*>(static_cast<const char*>(ws) + ws_o_bytes(B, Hq, D, S));
  c.seq_lens = lens;
  c.out = static_cast<uint16_t*>(out);
  c.out_stride = static_cast<int64_t>(Hq) * D;
  c.num_seqs = B;
  c.num_q_heads = Hq;
  c.block_size = bs;
  c.max_blocks_per_seq = mbs;
  c.num_splits = S;
  c.chunk = chunk_pages(page_span_max(mbs, bs, W), S);
  c.sliding_window = W;
  c.skip_direct = 0;
  c.plan_seg = nullptr;
  c.num_kv_heads = 0;
  c.out8 = nullptr;
  c.out_scale = 1.0f;
  return c;
}

// Bytes of K + V one (page, kv head) holds.
double page_head_bytes(int bs, int D, int kv_dtype) {
  const double elem = kv_dtype == PD_KV_BF16 ? 2.0 : (kv_dtype == PD_KV_FP8_E4M3 ? 1.0 : 0.5625);
  return static_cast<double>(bs) * 2.0 * D * elem;
}

// Shape-only split count: one CTA per (sequence, kv head, split) with about
// one wave of resident CTAs when every sequence is at its maximum length.
int plan_splits(int B, int Hkv, int mbs, int bs, int W, int num_sms, int ctas_per_sm) {
  const int span = page_span_max(mbs, bs, W);
  const int64_t units = static_cast<int64_t>(B > 0 ? B : 1) * (Hkv > 0 ? Hkv : 1);
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * ctas_per_sm;
  int64_t S = (slots + units / 2) / units;
  if (S > span) S = span;
  if (S < 1) S = 1;
  if (S > kMaxSplits) S = kMaxSplits;
  return static_cast<int>(S);
}

// Length-aware split count. For each candidate S it replays the launch in
// block order (kv head fastest, then split, then sequence) onto `slots`
// equal-bandwidth CTA slots, each CTA costing a fixed start-up equivalent of
// kCtaOverheadBytes plus its pages' bytes, and adds the partial-write and
// combine traffic of the splits that hold keys; the smallest estimated
// makespan wins (ties: fewer splits).
constexpr double kCtaOverheadBytes = 40.0 * 1024.0;
int plan_splits_lengths(const int32_t* lens, int B, int Hkv, int Hq, int mbs, int bs, int W,
                        int D, int kv_dtype, int num_sms, int ctas_per_sm,
                        double* best_estimate = nullptr) {
  const int span = page_span_max(mbs, bs, W);
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * ctas_per_sm;
  const double phb = page_head_bytes(bs, D, kv_dtype);
  std::vector<int> P(B);
  const int cap = mbs * bs;
  for (int b = 0; b < B; ++b) {
    const int L = lens[b] < 0 ? 0 : (lens[b] > cap ? cap : lens[b]);
    P[b] = num_key_pages(L, W, bs);
  }
  int best_S = 1;
  double best_t = 1e300;
  std::vector<double> heap;
  const int max_S = span < kMaxSplits ? span : kMaxSplits;
  // candidates: 1..32, a geometric ladder above, and the split counts that
  // fill one to four waves of resident CTAs exactly
  std::vector<int> cand;
  for (int S = 1; S <= max_S; S = (S < 32 ? S + 1 : S + S / 8)) cand.push_back(S);
  const int64_t units = static_cast<int64_t>(B) * Hkv;
  for (int k = 1; k <= 4; ++k) {
    const int64_t w = k * slots / (units > 0 ? units : 1);
    for (int64_t S = w - 1; S <= w + 1; ++S)
      if (S >= 1 && S <= max_S) cand.push_back(static_cast<int>(S));
  }
  std::sort(cand.begin(), cand.end());
  cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
  for (const int S : cand) {
    const int chunk = chunk_pages(span, S);
    heap.assign(static_cast<size_t>(slots), 0.0);  // min-heap of slot free times
    double partial_bytes = 0.0;
    for (int b = 0; b < B; ++b) {
      const int n = (P[b] + chunk - 1) / chunk;
      for (int sp = 0; sp < n; ++sp) {
        const int pages = (sp == n - 1) ? P[b] - sp * chunk : chunk;
        const double cost = kCtaOverheadBytes + pages * phb;
        for (int g = 0; g < Hkv; ++g) {
          std::pop_heap(heap.begin(), heap.end(), std::greater<double>());
          heap.back() += cost;
          std::push_heap(heap.begin(), heap.end(), std::greater<double>());
        }
      }
      if (n > 1) partial_bytes += 2.0 * n * static_cast<double>(Hq / Hkv) * Hkv * (D + 2) * 4.0;
    }
    const double span_t = *std::max_element(heap.begin(), heap.end());
    const double t = span_t + partial_bytes / static_cast<double>(slots);
    if (t < best_t * (1.0 - 1e-9)) {
      best_t = t;
      best_S = S;
    }
  }
  if (best_estimate) *best_estimate = best_t;
  return best_S;
}

// ---------------------------------------------------------------------------
// Balanced plan. Layout, in int32 words from a 16-byte aligned base:
//   [0..8)                       header: magic, num_ctas, num_pieces, num_seqs,
//                                num_kv_heads, block_size, sliding_window,
//                                max_blocks_per_seq
//   [8, 8 + num_ctas + 1)        cta_begin: CTA c owns pieces [cta_begin[c], cta_begin[c+1])
//   [pieces_off, +4*num_pieces)  pieces: (sequence * Hkv + kv head, first key,
//                                end key, flags; bit 0: the only piece of its head)
//   [seg_off, +2*B*Hkv)          per (sequence, kv head): first piece, piece count
constexpr int32_t kPlanMagic = 0x50444231;  // "PDB1"
constexpr int kMaxBalancedCtas = 1024;      // also bounds the pieces of one head (combine)
struct PlanLayout {
  int64_t cta_off, pieces_off, seg_off, words;
};
PlanLayout plan_layout(int64_t num_ctas, int64_t num_pieces, int64_t segs) {
  PlanLayout l;
  l.cta_off = 8;
  l.pieces_off = (l.cta_off + num_ctas + 1 + 3) / 4 * 4;
  l.seg_off = l.pieces_off + 4 * num_pieces;
  l.words = l.seg_off + 2 * segs;
  return l;
}
int64_t balanced_max_ctas(int num_sms) {
  const int64_t n = static_cast<int64_t>(num_sms) * 4;  // at most 4 resident CTAs per SM
  return n < kMaxBalancedCtas ? n : kMaxBalancedCtas;
}
size_t balanced_ws_bytes(int64_t num_pieces, int G, int D) {
  const size_t o = (static_cast<size_t>(num_pieces) * G * D * sizeof(float) + 255) / 256 * 256;
  const size_t ml = (static_cast<size_t>(num_pieces) * G * 2 * sizeof(float) + 255) / 256 * 256;
  return o + ml;
}

// Cost of a piece boundary inside a share, in keys: a piece ends in a partly
// filled 64-key tile (half a tile on average) and adds a merge and a q load.
// Measured: a CTA's time grows by about 1 us per extra piece, which is what
// 2 to 3 pages of 16 rows take at every cache form's rate.
constexpr int kPieceCostKeys = 40;

// Cut the line of (sequence, kv head) key-page ranges, laid end to end in
// sequence-major order, into num_ctas shares of equal cost (page
// granularity); every share that crosses a range boundary becomes several
// pieces. The cost of a share is its pages plus kPieceCostKeys for each range
// boundary inside it: the cut runs on a virtual line (1/16 page units) with a
// gap of that cost after every range, so a share that takes in a boundary
// gets correspondingly fewer pages. (The gap is dropped when shares are only
// a few pages long, so that no share falls into a gap.)
int build_balanced_plan(const int32_t* lens, int B, int Hq, int Hkv, int D, int bs, int mbs,
                        int W, int kv_dtype, int num_sms, int32_t* plan, size_t plan_bytes,
                        int32_t* out_ctas, int32_t* out_pieces, size_t* out_ws) {
  const int G = Hq / Hkv;
  const int cap = mbs * bs;
  std::vector<int> L(B), P(B);
  int64_t T = 0;
  for (int b = 0; b < B; ++b) {
    L[b] = lens[b] < 0 ? 0 : (lens[b] > cap ? cap : lens[b]);
    P[b] = num_key_pages(L[b], W, bs);
    T += static_cast<int64_t>(P[b]) * Hkv;
  }
  int64_t NC = static_cast<int64_t>(num_sms) * balanced_ctas_per_sm(kv_dtype, D, G);
  if (NC > kMaxBalancedCtas) NC = kMaxBalancedCtas;
  if (NC > T) NC = T;
  const int64_t segs = static_cast<int64_t>(B) * Hkv;
  // the virtual line: 16 units per page, a gap after every non-empty range
  constexpr int64_t kU = 16;
  int64_t ranges = 0;
  for (int b = 0; b < B; ++b) ranges += P[b] > 0 ? Hkv : 0;
  int64_t gap = (kPieceCostKeys * kU + bs / 2) / bs;
  if (NC == 0 || T * kU < 4 * gap * NC) gap = 0;
  const int64_t VT = T * kU + gap * (ranges > 0 ? ranges - 1 : 0);
  // pieces: one per range, plus one per share boundary strictly inside a range
  std::vector<int32_t> pieces;
  std::vector<int32_t> cta_begin(NC + 1, 0);
  std::vector<int32_t> seg(2 * segs, 0);
  pieces.reserve(4 * (segs + NC));
  auto bound = [&](int64_t c) { return NC > 0 ? c * VT / NC : 0; };  // share c starts here
  int64_t pos = 0;  // virtual position of the current range's first page
  int64_t c = 0;    // share holding `pos`
  int64_t np = 0;
  for (int b = 0; b < B; ++b) {
    const int lo = window_lo(L[b], W);
    const int page0 = lo / bs;  // the sequence's first key page
    for (int g = 0; g < Hkv; ++g) {
      const int64_t sid = static_cast<int64_t>(b) * Hkv + g;
      seg[2 * sid] = static_cast<int32_t>(np);
      if (P[b] == 0) continue;
      int64_t a = 0;  // pages of this range already cut
      while (a < P[b]) {
        while (c + 1 < NC && bound(c + 1) <= pos + a * kU) {
          ++c;
          cta_begin[c] = static_cast<int32_t>(np);
        }
        // the pages whose virtual start lies before the next share's start
        const int64_t next = c + 1 < NC ? bound(c + 1) : VT;
        const int64_t e = std::min<int64_t>(P[b], (next - pos + kU - 1) / kU);
        const int t_begin = std::max(lo, static_cast<int>((page0 + a) * bs));
        const int t_end = std::min(L[b], static_cast<int>((page0 + e) * bs));
        pieces.push_back(static_cast<int32_t>(sid));
        pieces.push_back(t_begin);
        pieces.push_back(t_end);
        pieces.push_back(0);
        ++np;
        a = e;
      }
      const int32_t count = static_cast<int32_t>(np) - seg[2 * sid];
      seg[2 * sid + 1] = count;
      if (count == 1) pieces[4 * (np - 1) + 3] = 1;  // its head's only piece: write out
      pos += P[b] * kU + gap;
    }
  }
  for (int64_t k = c + 1; k <= NC; ++k) cta_begin[k] = static_cast<int32_t>(np);
  const PlanLayout lay = plan_layout(NC, np, segs);
  if (plan_bytes < static_cast<size_t>(lay.words) * 4) return PD_ERR_WORKSPACE_TOO_SMALL;
  plan[0] = kPlanMagic;
  plan[1] = static_cast<int32_t>(NC);
  plan[2] = static_cast<int32_t>(np);
  plan[3] = B;
  plan[4] = Hkv;
  plan[5] = bs;
  plan[6] = W;
  plan[7] = mbs;
  for (int64_t k = 0; k <= NC; ++k) plan[lay.cta_off + k] = cta_begin[k];
  for (int64_t k = lay.cta_off + NC + 1; k < lay.pieces_off; ++k) plan[k] = 0;
  std::copy(pieces.begin(), pieces.end(), plan + lay.pieces_off);
  std::copy(seg.begin(), seg.end(), plan + lay.seg_off);
  *out_ctas = static_cast<int32_t>(NC);
  *out_pieces = static_cast<int32_t>(np);
  *out_ws = balanced_ws_bytes(np, G, D);
  return PD_OK;
}

// Balanced schedule vs split schedule, both in the split planner's units
// (bytes one CTA slot streams): the balanced kernel gives every CTA the same
// pages, at a per-tile premium (its piece bookkeeping), one CTA start-up
// like any CTA, and a switch-over cost per extra piece; the split schedule's
// estimate is the planner's best makespan. The premiums, 8 % (head_dim <=
// 128) and 12 % (head_dim 256 / 512, whose consumer warps also meet at a
// barrier every tile), are the ones that order the bench workloads as
// measured (equal lengths: split; unequal: balanced).
constexpr double kBalancedTilePremium = 1.08;
constexpr double kBalancedTilePremiumSplitD = 1.12;
constexpr double kPieceOverheadBytes = 8.0 * 1024.0;
int prefer_balanced(const int32_t* lens, int B, int Hq, int Hkv, int mbs, int bs, int W, int D,
                    int kv_dtype, int num_sms) {
  double split_t = 0.0;
  plan_splits_lengths(lens, B, Hkv, Hq, mbs, bs, W, D, kv_dtype, num_sms,
                      mma_ctas_per_sm_estimate(kv_dtype, D), &split_t);
  const int cap = mbs * bs;
  int64_t T = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lens[b] < 0 ? 0 : (lens[b] > cap ? cap : lens[b]);
    T += static_cast<int64_t>(num_key_pages(L, W, bs)) * Hkv;
  }
  if (T == 0) return 0;
  int64_t NC = static_cast<int64_t>(num_sms) * balanced_ctas_per_sm(kv_dtype, D, Hq / Hkv);
  if (NC > kMaxBalancedCtas) NC = kMaxBalancedCtas;
  if (NC > T) NC = T;
  const double pieces_per_cta = static_cast<double>(static_cast<int64_t>(B) * Hkv + NC) / NC;
  const double premium = D <= 128 ? kBalancedTilePremium : kBalancedTilePremiumSplitD;
  const double bal_t = premium * T * page_head_bytes(bs, D, kv_dtype) / NC +
                       kCtaOverheadBytes + (pieces_per_cta - 1.0) * kPieceOverheadBytes;
  return bal_t < split_t ? 1 : 0;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PD_OK : PD_ERR_CUDA; }

// A q row stride (elements between consecutive sequences' q rows): 0 means
// packed (Hq * D); otherwise at least Hq * D and a multiple of 8 elements so
// that every row starts on a 16-byte boundary.
bool q_stride_ok(int64_t q_stride, int Hq, int D) {
  return q_stride == 0 || (q_stride >= static_cast<int64_t>(Hq) * D && q_stride % 8 == 0);
}

}  // namespace

int decode_checks(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* seq_lens, const void* out,
                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                  int32_t num_splits, int32_t sliding_window, int32_t kv_dtype, float k_scale,
                  float v_scale, int64_t q_stride, int64_t out_stride, int* num_splits_out) {
  if (!q_stride_ok(q_stride, num_q_heads, head_dim)) return PD_ERR_INVALID_ARG;
  if (!q_stride_ok(out_stride, num_q_heads, head_dim)) return PD_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return PD_ERR_INVALID_ARG;
  // shapes first, so that a malformed request is refused before any CUDA call
  const DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_blocks_per_seq, 1, sliding_window, kv_dtype, num_blocks};
  const int rc = check_decode_shape(sh, k_scale, v_scale);
  if (rc != PD_OK) return rc;
  if (!isfinite(scale)) return PD_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!dev_ptr_ok(q) || !dev_ptr_ok(k_cache) || !dev_ptr_ok(v_cache) ||
                       !dev_ptr_ok(block_tables) || !dev_ptr_ok(seq_lens) || !dev_ptr_ok(out)))
    return PD_ERR_INVALID_ARG;
  int S = num_splits;
  if (S == 0) {
    DeviceInfo* dev = nullptr;
    if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
    S = plan_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, sliding_window,
                    dev->num_sms, mma_ctas_per_sm_estimate(kv_dtype, head_dim));
  }
  *num_splits_out = S;
  return PD_OK;
}

}  // namespace pd

using namespace pd;

extern "C" {

const char* pd_status_string(int status) {
  switch (status) {
    case PD_OK: return "PD_OK";
    case PD_ERR_INVALID_ARG: return "PD_ERR_INVALID_ARG: invalid argument";
    case PD_ERR_UNSUPPORTED: return "PD_ERR_UNSUPPORTED: unsupported shape or dtype";
    case PD_ERR_WORKSPACE_TOO_SMALL: return "PD_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case PD_ERR_CUDA: return "PD_ERR_CUDA: CUDA runtime error";
    default: return "unknown pd status";
  }
}

size_t pd_page_bytes(int32_t kv_dtype, int32_t block_size, int32_t num_kv_heads,
                     int32_t head_dim) {
  if (!dtype_ok(kv_dtype) || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (kv_dtype == PD_KV_NVFP4 && head_dim % 16 != 0) return 0;
  return static_cast<size_t>(page_bytes_of(kv_dtype, block_size, num_kv_heads, head_dim));
}

size_t pd_cache_bytes(int32_t kv_dtype, int64_t num_blocks, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_dim) {
  if (num_blocks < 0) return 0;
  return static_cast<size_t>(num_blocks) * pd_page_bytes(kv_dtype, block_size, num_kv_heads,
                                                         head_dim);
}

size_t pd_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t num_splits) {
  if (num_seqs < 0 || num_q_heads < 0 || head_dim < 0 || num_splits < 0) return 0;
  return ws_total_bytes(num_seqs, num_q_heads, head_dim, num_splits);
}

int pd_plan_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                       int32_t block_size, int32_t sliding_window, int32_t head_dim,
                       int32_t kv_dtype, int32_t num_sms) {
  if (num_seqs < 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
      sliding_window < 0 || num_sms <= 0 || !head_dim_ok(head_dim) || !dtype_ok(kv_dtype))
    return -PD_ERR_INVALID_ARG;
  return plan_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, sliding_window,
                     num_sms, mma_ctas_per_sm_estimate(kv_dtype, head_dim));
}

int pd_plan_num_splits_for_lengths(const int32_t* seq_lens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t max_blocks_per_seq, int32_t block_size,
                                   int32_t sliding_window, int32_t head_dim, int32_t kv_dtype,
                                   int32_t num_sms) {
  if (num_seqs < 0 || (num_seqs > 0 && seq_lens == nullptr) || num_kv_heads <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0 || sliding_window < 0 || num_sms <= 0 || !head_dim_ok(head_dim) ||
      !dtype_ok(kv_dtype))
    return -PD_ERR_INVALID_ARG;
  if (num_seqs == 0) return 1;
  return plan_splits_lengths(seq_lens, num_seqs, num_kv_heads, num_q_heads, max_blocks_per_seq,
                             block_size, sliding_window, head_dim, kv_dtype, num_sms,
                             mma_ctas_per_sm_estimate(kv_dtype, head_dim));
}

int pd_choose_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                         int32_t block_size, int32_t sliding_window, int32_t head_dim,
                         int32_t kv_dtype, int device) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return -PD_ERR_CUDA;
  return pd_plan_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size,
                            sliding_window, head_dim, kv_dtype, sms);
}

int pd_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int32_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         int32_t kv_dtype, float k_scale, float v_scale, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PD_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size) || !dtype_ok(kv_dtype))
    return PD_ERR_UNSUPPORTED;
  if (kv_dtype == PD_KV_FP8_E4M3 && !(scale_ok(k_scale) && scale_ok(v_scale)))
    return PD_ERR_INVALID_ARG;
  if (num_tokens == 0) return PD_OK;
  if (!dev_ptr_ok(key) || !dev_ptr_ok(value) || !dev_ptr_ok(k_cache) || !dev_ptr_ok(v_cache) ||
      !dev_ptr_ok(slot_mapping))
    return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  return cuda_status(launch_reshape_and_cache(
      static_cast<const uint16_t*>(key), static_cast<const uint16_t*>(value),
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), slot_mapping, num_tokens,
      num_kv_heads, head_dim, block_size, num_blocks, kv_dtype, k_scale, v_scale, dev->flags,
      static_cast<cudaStream_t>(stream)));
}

int pd_absmax_bf16(const void* data, int64_t n, float* out_max, void* stream) {
  if (n < 0) return PD_ERR_INVALID_ARG;
  if (n == 0) return PD_OK;
  if (!dev_ptr_ok(data) || out_max == nullptr || (reinterpret_cast<uintptr_t>(out_max) & 3u))
    return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  return cuda_status(launch_absmax(static_cast<const uint16_t*>(data), n, out_max, dev->num_sms,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
int partial_impl(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                 int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t num_splits,
                 int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                 void* workspace, size_t workspace_bytes, void* stream, int64_t q_stride,
                 bool cuda_core = false) {
  const DecodeShape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_splits, sliding_window, kv_dtype, num_blocks};
  const int rc = check_decode(s, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                              workspace, workspace_bytes);
  if (rc != PD_OK || num_seqs == 0) return rc;
  if (!isfinite(scale)) return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  DecodeArgs a = make_decode_args(s, q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale,
                                  v_scale, workspace, dev->flags);
  if (!q_stride_ok(q_stride, num_q_heads, head_dim)) return PD_ERR_INVALID_ARG;
  if (q_stride) a.q_stride = q_stride;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(cuda_core ? launch_decode_partial(a, head_dim, kv_dtype, st)
                               : launch_decode_partial_mma(a, head_dim, kv_dtype, st));
}
}  // namespace

extern "C" {

int pd_decode_partial(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks,
                      float scale, int32_t num_splits, int32_t sliding_window, int32_t kv_dtype,
                      float k_scale, float v_scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return partial_impl(q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                      num_splits, sliding_window, kv_dtype, k_scale, v_scale, workspace,
                      workspace_bytes, stream, 0);
}

int pd_decode_combine(const void* workspace, size_t workspace_bytes, const int32_t* seq_lens,
                      void* out, int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_blocks_per_seq, int32_t num_splits,
                      int32_t sliding_window, void* stream) {
  if (num_seqs < 0 || num_seqs > 65535 || num_q_heads <= 0 || max_blocks_per_seq <= 0 ||
      sliding_window < 0 || num_splits < 1 || num_splits > kMaxSplits)
    return PD_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PD_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PD_OK;
  if (!dev_ptr_ok(workspace) || !dev_ptr_ok(seq_lens) || !dev_ptr_ok(out))
    return PD_ERR_INVALID_ARG;
  if (workspace_bytes < ws_total_bytes(num_seqs, num_q_heads, head_dim, num_splits))
    return PD_ERR_WORKSPACE_TOO_SMALL;
  const CombineArgs c = make_combine_args(num_seqs, num_q_heads, head_dim, block_size,
                                          max_blocks_per_seq, num_splits, sliding_window,
                                          workspace, seq_lens, out);
  return cuda_status(
      launch_decode_combine(c, head_dim, num_splits, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
int decode_split(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* seq_lens, void* out,
                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                 int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                 int32_t num_splits, int32_t sliding_window, int32_t kv_dtype, float k_scale,
                 float v_scale, void* workspace, size_t workspace_bytes, void* stream,
                 int64_t q_stride, int64_t out_stride = 0, bool cuda_core = false,
                 float e4m3_out_scale = 0.0f) {
  int S = 0;
  const int rc = decode_checks(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs,
                               num_q_heads, num_kv_heads, head_dim, block_size,
                               max_blocks_per_seq, num_blocks, scale, num_splits, sliding_window,
                               kv_dtype, k_scale, v_scale, q_stride, out_stride, &S);
  if (rc != PD_OK || num_seqs == 0) return rc;
  if (!dev_ptr_ok(workspace)) return PD_ERR_INVALID_ARG;
  if (workspace_bytes < ws_total_bytes(num_seqs, num_q_heads, head_dim, S))
    return PD_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  const DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_blocks_per_seq, S, sliding_window, kv_dtype, num_blocks};
  DecodeArgs a = make_decode_args(sh, q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale,
                                  v_scale, workspace, dev->flags);
  if (q_stride) a.q_stride = q_stride;
  if (out_stride) a.out_stride = out_stride;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  CombineArgs c = make_combine_args(num_seqs, num_q_heads, head_dim, block_size,
                                    max_blocks_per_seq, S, sliding_window, workspace, seq_lens,
                                    out);
  if (out_stride) c.out_stride = out_stride;
  if (e4m3_out_scale > 0.0f) {
    // E4M3 output: every sequence's partials go through the workspace and the
    // combine writes the codes
    c.out = nullptr;
    c.out8 = static_cast<uint8_t*>(out);
    c.out_scale = e4m3_out_scale;
    const cudaError_t e = cuda_core ? launch_decode_partial(a, head_dim, kv_dtype, st)
                                    : launch_decode_partial_mma(a, head_dim, kv_dtype, st);
    if (e != cudaSuccess) return PD_ERR_CUDA;
    return cuda_status(launch_decode_combine(c, head_dim, S, st));
  }
  if (cuda_core) {
    // the CUDA-core cross-check kernel writes every partial; the combine merges all
    if (launch_decode_partial(a, head_dim, kv_dtype, st) != cudaSuccess) return PD_ERR_CUDA;
    return cuda_status(launch_decode_combine(c, head_dim, S, st));
  }
  // the partial kernel writes the rows of sequences whose keys fit one split
  // (and zero rows for empty ones); the combine merges the rest
  a.out = static_cast<uint16_t*>(out);
  a.direct = 1;
  if (launch_decode_partial_mma(a, head_dim, kv_dtype, st) != cudaSuccess) return PD_ERR_CUDA;
  c.skip_direct = 1;
  return cuda_status(launch_decode_combine(c, head_dim, S, st));
}
}  // namespace

extern "C" {

int pd_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* seq_lens, void* out, int32_t num_seqs, int32_t num_q_heads,
              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
              int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t num_splits,
              int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
              void* workspace, size_t workspace_bytes, void* stream) {
  return decode_split(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                      num_splits, sliding_window, kv_dtype, k_scale, v_scale, workspace,
                      workspace_bytes, stream, 0);
}

int pd_decode_strided(const void* q, int64_t q_stride, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, void* out,
                      int64_t out_stride, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                      int32_t num_splits, int32_t sliding_window, int32_t kv_dtype,
                      float k_scale, float v_scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (q_stride <= 0 || out_stride <= 0) return PD_ERR_INVALID_ARG;
  return decode_split(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                      num_splits, sliding_window, kv_dtype, k_scale, v_scale, workspace,
                      workspace_bytes, stream, q_stride, out_stride);
}

int pd_prefer_balanced(const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t max_blocks_per_seq, int32_t block_size,
                       int32_t sliding_window, int32_t head_dim, int32_t kv_dtype,
                       int32_t num_sms) {
  if (num_seqs < 0 || (num_seqs > 0 && seq_lens == nullptr) || num_kv_heads <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0 || sliding_window < 0 || num_sms <= 0 || !head_dim_ok(head_dim) ||
      !dtype_ok(kv_dtype) || num_q_heads / num_kv_heads > kMaxGroup)
    return -PD_ERR_INVALID_ARG;
  if (num_seqs == 0) return 0;
  return prefer_balanced(seq_lens, num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq,
                         block_size, sliding_window, head_dim, kv_dtype, num_sms);
}

size_t pd_balanced_plan_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t num_sms) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_sms <= 0) return 0;
  const int64_t nc = balanced_max_ctas(num_sms);
  const int64_t segs = static_cast<int64_t>(num_seqs) * num_kv_heads;
  return static_cast<size_t>(plan_layout(nc, segs + nc, segs).words) * 4;
}

int pd_balanced_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t max_blocks_per_seq, int32_t sliding_window, int32_t kv_dtype,
                     int32_t num_sms, void* plan, size_t plan_bytes, int32_t* num_ctas,
                     int32_t* num_pieces, size_t* workspace_bytes) {
  if (num_seqs < 0 || num_seqs > 65535 || (num_seqs > 0 && seq_lens == nullptr) ||
      num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      max_blocks_per_seq <= 0 || sliding_window < 0 || num_sms <= 0 || plan == nullptr ||
      (reinterpret_cast<uintptr_t>(plan) & 15u) || num_ctas == nullptr ||
      num_pieces == nullptr || workspace_bytes == nullptr)
    return PD_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > kMaxGroup) return PD_ERR_UNSUPPORTED;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size) || !dtype_ok(kv_dtype))
    return PD_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > (int64_t{1} << 30))
    return PD_ERR_INVALID_ARG;
  return build_balanced_plan(seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, sliding_window, kv_dtype, num_sms,
                             static_cast<int32_t*>(plan), plan_bytes, num_ctas, num_pieces,
                             workspace_bytes);
}

}  // extern "C"

namespace {
// pd_decode_balanced and its two halves: which of the two kernels to launch.
int decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const void* plan, size_t plan_bytes, void* out,
                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                    int64_t num_blocks, float scale, int32_t sliding_window, int32_t kv_dtype,
                    float k_scale, float v_scale, int32_t num_ctas, int32_t num_pieces,
                    void* workspace, size_t workspace_bytes, void* stream, bool partial,
                    bool combine, int64_t q_stride = 0, int64_t out_stride = 0) {
  if (!q_stride_ok(q_stride, num_q_heads, head_dim)) return PD_ERR_INVALID_ARG;
  if (!q_stride_ok(out_stride, num_q_heads, head_dim)) return PD_ERR_INVALID_ARG;
  // shape checks shared with pd_decode (S = 1 stands for the split count)
  const DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_blocks_per_seq, 1, sliding_window, kv_dtype, num_blocks};
  if (num_ctas < 0 || num_ctas > kMaxBalancedCtas || num_pieces < 0 ||
      (num_ctas == 0) != (num_pieces == 0))
    return PD_ERR_INVALID_ARG;
  const int64_t segs = static_cast<int64_t>(num_seqs) * (num_kv_heads > 0 ? num_kv_heads : 0);
  if (static_cast<int64_t>(num_pieces) > segs + num_ctas) return PD_ERR_INVALID_ARG;
  int rc = check_decode(sh, q, k_cache, v_cache, block_tables, block_tables, k_scale, v_scale,
                        workspace, SIZE_MAX);
  if (rc != PD_OK || num_seqs == 0) return rc;
  if (!isfinite(scale) || !dev_ptr_ok(out) || !dev_ptr_ok(plan)) return PD_ERR_INVALID_ARG;
  const PlanLayout lay = plan_layout(num_ctas, num_pieces, segs);
  if (plan_bytes < static_cast<size_t>(lay.words) * 4) return PD_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (workspace_bytes < balanced_ws_bytes(num_pieces, G, head_dim))
    return PD_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  const int32_t* pl = static_cast<const int32_t*>(plan);
  DecodeArgs a = make_decode_args(sh, q, k_cache, v_cache, block_tables, nullptr, scale, k_scale,
                                  v_scale, workspace, dev->flags);
  // balanced workspace: O [pieces][G][D], then (m, l) [pieces][G]
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = reinterpret_cast<float2*>(
      static_cast<char*>(workspace) +
      (static_cast<size_t>(num_pieces) * G * head_dim * sizeof(float) + 255) / 256 * 256);
  a.out = static_cast<uint16_t*>(out);
  a.direct = 1;
  a.plan_cta = pl + lay.cta_off;
  a.plan_pieces = reinterpret_cast<const int4*>(pl + lay.pieces_off);
  a.plan_num_ctas = num_ctas;
  a.plan_num_pieces = num_pieces;
  if (q_stride) a.q_stride = q_stride;
  if (out_stride) a.out_stride = out_stride;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (partial && launch_decode_partial_balanced(a, head_dim, kv_dtype, st) != cudaSuccess)
    return PD_ERR_CUDA;
  if (!combine) return PD_OK;
  CombineArgs c = make_combine_args(num_seqs, num_q_heads, head_dim, block_size,
                                    max_blocks_per_seq, 1, sliding_window, workspace, nullptr,
                                    out);
  c.ws_o = a.ws_o;
  c.ws_ml = a.ws_ml;
  c.plan_seg = pl + lay.seg_off;
  c.num_kv_heads = num_kv_heads;
  if (out_stride) c.out_stride = out_stride;
  // a (sequence, kv head) range has ceil(pieces / ranges) pieces on average;
  // the plan's longest may have more (its rows then take a few more loads)
  const int64_t avg = segs > 0 ? (num_pieces + segs - 1) / segs : 1;
  return cuda_status(launch_decode_combine(c, head_dim, static_cast<int>(avg), st));
}
}  // namespace

extern "C" {

int pd_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const void* plan, size_t plan_bytes,
                       void* out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                       int64_t num_blocks, float scale, int32_t sliding_window,
                       int32_t kv_dtype, float k_scale, float v_scale, int32_t num_ctas,
                       int32_t num_pieces, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return decode_balanced(q, k_cache, v_cache, block_tables, plan, plan_bytes, out, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         num_blocks, scale, sliding_window, kv_dtype, k_scale, v_scale, num_ctas,
                         num_pieces, workspace, workspace_bytes, stream, true, true);
}

int pd_decode_balanced_strided(const void* q, int64_t q_stride, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const void* plan, size_t plan_bytes, void* out,
                               int64_t out_stride, int32_t num_seqs,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, int32_t sliding_window,
                               int32_t kv_dtype, float k_scale, float v_scale, int32_t num_ctas,
                               int32_t num_pieces, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (q_stride <= 0 || out_stride <= 0) return PD_ERR_INVALID_ARG;
  return decode_balanced(q, k_cache, v_cache, block_tables, plan, plan_bytes, out, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         num_blocks, scale, sliding_window, kv_dtype, k_scale, v_scale, num_ctas,
                         num_pieces, workspace, workspace_bytes, stream, true, true, q_stride,
                         out_stride);
}

int pd_decode_balanced_partial(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const void* plan, size_t plan_bytes,
                               void* out, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                               int32_t sliding_window, int32_t kv_dtype, float k_scale,
                               float v_scale, int32_t num_ctas, int32_t num_pieces,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_balanced(q, k_cache, v_cache, block_tables, plan, plan_bytes, out, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         num_blocks, scale, sliding_window, kv_dtype, k_scale, v_scale, num_ctas,
                         num_pieces, workspace, workspace_bytes, stream, true, false);
}

int pd_decode_balanced_combine(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const void* plan, size_t plan_bytes,
                               void* out, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                               int32_t sliding_window, int32_t kv_dtype, float k_scale,
                               float v_scale, int32_t num_ctas, int32_t num_pieces,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_balanced(q, k_cache, v_cache, block_tables, plan, plan_bytes, out, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         num_blocks, scale, sliding_window, kv_dtype, k_scale, v_scale, num_ctas,
                         num_pieces, workspace, workspace_bytes, stream, false, true);
}

}  // extern "C"

namespace {
int prefill_impl(const void* q, int64_t q_stride, const int32_t* cu_q, const void* k_cache,
                 const void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                 void* out, int64_t out_stride, int32_t num_seqs, int32_t max_q_len,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                 int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t causal,
                 int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                 void* stream, bool mma_sync) {
  if (num_seqs < 0 || num_seqs > 65535 || max_q_len < 0) return PD_ERR_INVALID_ARG;
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return PD_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (G > kMaxGroup || num_kv_heads > 65535) return PD_ERR_UNSUPPORTED;
  if (!dtype_ok(kv_dtype) || !head_dim_ok(head_dim) || !block_size_ok(block_size))
    return PD_ERR_UNSUPPORTED;
  if (head_dim > 256) return PD_ERR_UNSUPPORTED;
  if (kv_dtype == PD_KV_FP8_E4M3 && !(scale_ok(k_scale) && scale_ok(v_scale)))
    return PD_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 || sliding_window < 0) return PD_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > (int64_t{1} << 30))
    return PD_ERR_INVALID_ARG;
  if (num_blocks * block_size > INT32_MAX) return PD_ERR_INVALID_ARG;
  if (!q_stride_ok(q_stride, num_q_heads, head_dim) || !q_stride_ok(out_stride, num_q_heads, head_dim))
    return PD_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PD_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_q_len == 0) return PD_OK;
  if (!dev_ptr_ok(q) || !dev_ptr_ok(cu_q) || !dev_ptr_ok(k_cache) || !dev_ptr_ok(v_cache) ||
      !dev_ptr_ok(block_tables) || !dev_ptr_ok(seq_lens) || !dev_ptr_ok(out))
    return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  PrefillArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.q_stride = q_stride ? q_stride : static_cast<int64_t>(num_q_heads) * head_dim;
  a.cu_q = cu_q;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.out = static_cast<uint16_t*>(out);
  a.out_stride = out_stride ? out_stride : static_cast<int64_t>(num_q_heads) * head_dim;
  a.flags = dev->flags;
  a.num_blocks = num_blocks;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = G;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.causal = causal != 0;
  a.sliding_window = sliding_window;
  a.scale_log2 = scale * kLog2e;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the tcgen05 kernel reads BF16 caches; FP8 / NVFP4 caches (and the
  // cross-check) run on the mma.sync kernel, which widens each stage to f16
  if (mma_sync || kv_dtype != PD_KV_BF16) {
    a.tokens_per_cta = 64 / G;
    return cuda_status(launch_prefill(a, k_cache, v_cache, head_dim, kv_dtype, max_q_len, st));
  }
  a.tokens_per_cta = 128 / G;
  if (head_dim <= 128)
    return cuda_status(launch_prefill_pair(a, k_cache, v_cache, head_dim, max_q_len, st));
  return cuda_status(launch_prefill_umma(a, k_cache, v_cache, head_dim, max_q_len, st));
}

}  // namespace

extern "C" {

int pd_prefill(const void* q, int64_t q_stride, const int32_t* cu_q, const void* k_cache,
               const void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
               void* out, int64_t out_stride, int32_t num_seqs, int32_t max_q_len,
               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
               int32_t max_blocks_per_seq, int64_t num_blocks, float scale, int32_t causal,
               int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
               void* stream) {
  return prefill_impl(q, q_stride, cu_q, k_cache, v_cache, block_tables, seq_lens, out,
                      out_stride, num_seqs, max_q_len, num_q_heads, num_kv_heads, head_dim,
                      block_size, max_blocks_per_seq, num_blocks, scale, causal, sliding_window,
                      kv_dtype, k_scale, v_scale, stream, false);
}

int pd_prefill_crosscheck(const void* q, int64_t q_stride, const int32_t* cu_q,
                          const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          const int32_t* seq_lens, void* out, int64_t out_stride,
                          int32_t num_seqs, int32_t max_q_len, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                          int32_t causal, int32_t sliding_window, int32_t kv_dtype,
                          float k_scale, float v_scale, void* stream) {
  return prefill_impl(q, q_stride, cu_q, k_cache, v_cache, block_tables, seq_lens, out,
                      out_stride, num_seqs, max_q_len, num_q_heads, num_kv_heads, head_dim,
                      block_size, max_blocks_per_seq, num_blocks, scale, causal, sliding_window,
                      kv_dtype, k_scale, v_scale, stream, true);
}

int pd_decode_crosscheck(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, void* out,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                         int64_t num_blocks, float scale, int32_t num_splits,
                         int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return decode_split(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                      num_splits, sliding_window, kv_dtype, k_scale, v_scale, workspace,
                      workspace_bytes, stream, 0, 0, true);
}

int pd_decode_e4m3_out(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens, void* out,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                       int64_t num_blocks, float scale, int32_t num_splits,
                       int32_t sliding_window, int32_t kv_dtype, float k_scale, float v_scale,
                       float out_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!(isfinite(out_scale) && out_scale > 0.0f)) return PD_ERR_INVALID_ARG;
  return decode_split(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                      num_splits, sliding_window, kv_dtype, k_scale, v_scale, workspace,
                      workspace_bytes, stream, 0, 0, false, out_scale);
}

float pd_fp8_scale(float absmax) { return absmax > 0.0f ? absmax / 448.0f : 1.0f; }

int pd_fp8_scales_from_absmax(const float* absmax, float* scales, int32_t count, void* stream) {
  if (count < 0) return PD_ERR_INVALID_ARG;
  if (count == 0) return PD_OK;
  const uintptr_t a = reinterpret_cast<uintptr_t>(absmax), o = reinterpret_cast<uintptr_t>(scales);
  if (absmax == nullptr || scales == nullptr || (a & 3u) || (o & 3u)) return PD_ERR_INVALID_ARG;
  return cuda_status(launch_fp8_scales(absmax, scales, count, static_cast<cudaStream_t>(stream)));
}

int pd_device_status(int32_t* flags, int32_t reset) {
  if (flags == nullptr) return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_flags, sizeof(int)) != cudaSuccess) return PD_ERR_CUDA;
  *flags = v;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_flags, &zero, sizeof(int)) != cudaSuccess) return PD_ERR_CUDA;
  }
  return PD_OK;
}

int pd_test_encode(int32_t format, uint32_t first_bits, int64_t count, uint8_t* codes,
                   void* stream) {
  if ((format != 0 && format != 1) || count < 0 || count > (int64_t{1} << 32))
    return PD_ERR_INVALID_ARG;
  if (count == 0) return PD_OK;
  if (codes == nullptr) return PD_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != cudaSuccess) return PD_ERR_CUDA;
  return cuda_status(launch_encode_bits(format, first_bits, count, codes, dev->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

uint32_t pd_test_set_consumer_wait_ns(uint32_t ns) {
  return g_consumer_wait_ns.exchange(ns == 0xFFFFFFFFu ? kDefaultConsumerWaitNs : ns);
}

}  // extern "C"
