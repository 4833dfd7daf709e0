// The per-tile work of the tensor-core partial kernels' consumer warps,
// shared by decode_mma.cu (one CTA per split) and decode_balanced.cu (one CTA
// per plan share): the q fragments of a GQA group, and for one stage of keys
// the scores S^T = K Q^T, one online-softmax update and O^T += V^T P^T on
// mma.sync, with keys on M and the group's q heads on N.
#pragma once

#include <type_traits>

#include "mma_common.cuh"

namespace pd {
namespace mma {

// A consumer thread's registers for one (sequence, kv head, key range): the q
// fragments (B operand of the scores) and their score multipliers, the O^T
// accumulator and the per-column running max and sum.
template <class C, int NT>
struct TileState {
  uint32_t qf[C::kKSteps][NT][2];
  float qmul[NT][2];  // score multiplier (log2 units) of the two head columns of this thread
  float acc[C::kKSteps][NT][4];  // O^T: [head_dim m-tile][n-tile][fragment]
  float m_run[NT][2], l_run[NT][2];
};

// The consumer thread's place: warp, lane, fragment row group r = lane / 4,
// column pair c = lane % 4, and the first head_dim index of its warp's slice.
struct ThreadPlace {
  int warp, lane, r, c, d0;
};

// One stage as the consumers see it: the K and V halves in shared memory, the
// key index of its first row, the key range [t_begin, t_end) that counts, and
// the copies whose pages were outside the pool (their keys are masked).
struct StageView {
  uint32_t kst, vst;
  int t0, t_begin, t_end;
  uint32_t bad;
};

// q fragments of the group's G heads from qb (G rows of D bf16, global or
// shared memory). BF16: natural order, k index = d. f16 forms: thread column
// c owns the slice's d in [c*DS/4, (c+1)*DS/4); k-step ks uses
// d = c*DS/4 + 4ks + {0..3}. head_dim split: the four consumer warps meet at
// named barrier 1 (their callers guarantee that all four get here).
template <int FMT, int D, int NT, class C>
__device__ __forceinline__ void load_q_fragments(TileState<C, NT>& s, const uint16_t* qb, int G,
                                                 float scale_log2, float k_scale,
                                                 const ThreadPlace& tp, float* qmax_s) {
  constexpr bool F16 = C::kF16;
  const int warp = tp.warp, r = tp.r, c = tp.c, d0 = tp.d0;
  auto& qf = s.qf;
  auto& qmul = s.qmul;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = nt * 8 + r;  // q head row of the B fragment
    if constexpr (!F16) {
      qmul[nt][0] = qmul[nt][1] = scale_log2;
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
        qmul[nt][j] = scale_log2 * (FMT == PD_KV_FP8_E4M3 ? k_scale : 1.0f) *
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

// Zero the running state for a new key range.
template <class C, int NT>
__device__ __forceinline__ void reset_state(TileState<C, NT>& s) {
#pragma unroll
  for (int i = 0; i < C::kKSteps; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) s.acc[i][nt][k] = 0.0f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s.m_run[nt][0] = s.m_run[nt][1] = -INFINITY;
    s.l_run[nt][0] = s.l_run[nt][1] = 0.0f;
  }
}

// One stage of keys into the running state. head_dim split: the warps sum
// their partial scores through `red` (buffer red_buf) at named barrier 1,
// which every consumer warp must reach.
template <int FMT, int D, int NT, class C>
__device__ __forceinline__ void consume_tile(TileState<C, NT>& s, const StageView& sv,
                                             const ThreadPlace& tp, const float* red_in,
                                             int red_buf) {
  constexpr bool F16 = C::kF16;
  const int warp = tp.warp, lane = tp.lane, r = tp.r, c = tp.c, d0 = tp.d0;
  const uint32_t kst = sv.kst, vst = sv.vst;
  const int t0 = sv.t0, t_begin = sv.t_begin, t_end = sv.t_end;
  const uint32_t bad = sv.bad;
  float* red = const_cast<float*>(red_in);
  auto& qf = s.qf;
  auto& qmul = s.qmul;
  auto& acc = s.acc;
  auto& m_run = s.m_run;
  auto& l_run = s.l_run;
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

}

}  // namespace mma
}  // namespace pd
