// Cache write / quantise (metrale "prefill_attn_b.rs", `reshape_and_cache_nvfp4`:
// one block per token writes its K and V rows at the slot_mapping slot) and the
// bf16 absmax used for FP8 calibration (same page, `bf16_absmax`).
#include "pd_common.cuh"

namespace pd {
namespace {

constexpr int kWriteThreads = 256;

// x / s with IEEE division (no fast-math reciprocal). A NaN x goes through
// unchanged: the GPU's NaN results are canonical (positive), and the code of
// a NaN input takes the input's own sign.
__device__ __forceinline__ float quotient(float x, float s) {
  return (x != x) ? x : __fdiv_rn(x, s);
}

// BF16: byte copy of the token's [Hkv][D] row into page slot/bs, row slot%bs.
__device__ __forceinline__ void copy_row_bf16(const uint16_t* src, uint8_t* dst, int row_elems) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < row_elems / 8; i += blockDim.x) d[i] = __ldg(s + i);
}

// FP8: 8 elements per thread, E4M3(float(x) / scale) with IEEE division.
__device__ __forceinline__ void quant_row_fp8(const uint16_t* src, uint8_t* dst, int row_elems,
                                              float scale) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint2* d = reinterpret_cast<uint2*>(dst);
  for (int i = threadIdx.x; i < row_elems / 8; i += blockDim.x) {
    const uint4 v = __ldg(s + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float x = (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]);
      const uint32_t c = e4m3_encode(quotient(x, scale));
      out[k >> 2] |= c << (8 * (k & 3));
    }
    d[i] = make_uint2(out[0], out[1]);
  }
}

// NVFP4: one 16-element group per thread: scale = E4M3(amax / 6), codes
// E2M1(x / decode(scale)), +0 codes when the scale decodes to zero.
__device__ __forceinline__ void quant_row_nvfp4(const uint16_t* src, uint8_t* page, int hkv, int d,
                                                int bs, int row, int64_t data_bytes) {
  const int groups_per_head = d / 16;
  for (int gi = threadIdx.x; gi < hkv * groups_per_head; gi += blockDim.x) {
    const int h = gi / groups_per_head;
    const int grp = gi % groups_per_head;
    const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(gi) * 16);
    const uint4 v0 = __ldg(s);
    const uint4 v1 = __ldg(s + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = bf16_lo(w[k]);
      x[2 * k + 1] = bf16_hi(w[k]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));  // fmaxf drops NaN
    const uint32_t sc = e4m3_encode(__fdiv_rn(amax, 6.0f));
    const float sdec = e4m3_decode(sc);
    uint32_t packed[2] = {0u, 0u};
    if (sdec != 0.0f) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint32_t c = e2m1_encode(quotient(x[k], sdec));
        packed[k >> 3] |= c << (4 * (k & 7));
      }
    }
    const int64_t line = static_cast<int64_t>(h) * bs + row;
    *reinterpret_cast<uint2*>(page + line * (d / 2) + grp * 8) = make_uint2(packed[0], packed[1]);
    page[data_bytes + line * groups_per_head + grp] = static_cast<uint8_t>(sc);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kWriteThreads)
    reshape_and_cache_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                             uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                             const int32_t* __restrict__ slots, int hkv, int d, int bs,
                             int64_t num_blocks, float k_scale, float v_scale, int64_t page_bytes,
                             int64_t data_bytes, int* flags) {
  // Launched as a programmatic dependent of the previous work on the stream
  // (the previous step's combine, say): nothing global is touched before that
  // grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_blocks * bs) {
    if (threadIdx.x == 0) atomicOr(flags, PD_DEV_BAD_SLOT);
    return;
  }
  const int64_t page = slot / bs;
  const int row = static_cast<int>(slot % bs);
  const int row_elems = hkv * d;
  const uint16_t* ksrc = key + static_cast<int64_t>(t) * row_elems;
  const uint16_t* vsrc = value + static_cast<int64_t>(t) * row_elems;
  uint8_t* kpage = k_cache + page * page_bytes;
  uint8_t* vpage = v_cache + page * page_bytes;
  if (FMT == PD_KV_BF16) {
    copy_row_bf16(ksrc, kpage + static_cast<int64_t>(row) * row_elems * 2, row_elems);
    copy_row_bf16(vsrc, vpage + static_cast<int64_t>(row) * row_elems * 2, row_elems);
  } else if (FMT == PD_KV_FP8_E4M3) {
    quant_row_fp8(ksrc, kpage + static_cast<int64_t>(row) * row_elems, row_elems, k_scale);
    quant_row_fp8(vsrc, vpage + static_cast<int64_t>(row) * row_elems, row_elems, v_scale);
  } else {
    quant_row_nvfp4(ksrc, kpage, hkv, d, bs, row, data_bytes);
    quant_row_nvfp4(vsrc, vpage, hkv, d, bs, row, data_bytes);
  }
  // the decode that reads these rows may now be placed; it still waits for
  // this grid's completion (griddepcontrol.wait) before its first read
  asm volatile("griddepcontrol.launch_dependents;");
}

// max |x| over bf16 values: grid-stride over 16-byte chunks, warp and block
// reductions, one atomicMax per block on the non-negative float's bits.
__global__ void __launch_bounds__(256)
    absmax_bf16_kernel(const uint16_t* __restrict__ data, int64_t n, float* out_max) {
  float m = 0.0f;
  const int64_t nvec = n / 8;
  const uint4* v = reinterpret_cast<const uint4*>(data);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += stride) {
    const uint4 w = __ldg(v + i);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = fmaxf(m, fabsf(bf16_lo(ws[k])));
      m = fmaxf(m, fabsf(bf16_hi(ws[k])));
    }
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    m = fmaxf(m, fabsf(bf16_to_f32(data[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (blockDim.x >> 5); ++k) m = fmaxf(m, wmax[k]);
    atomicMax(reinterpret_cast<int*>(out_max), __float_as_int(m));
  }
}

// FP8 calibration scales from absmax values: absmax / 448 with IEEE fp32
// division, 1 where the absmax is not positive (an all-zero tensor, or NaN).
__global__ void fp8_scales_kernel(const float* __restrict__ absmax, float* __restrict__ scales,
                                  int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const float a = absmax[i];
    scales[i] = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
  }
}

// The cache write's own encoders applied to fp32 bit patterns first + i
// (i < n): format 0 = E4M3, 1 = E2M1 (one code per byte).
__global__ void encode_bits_kernel(int format, uint32_t first, int64_t n, uint8_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float x = __uint_as_float(first + static_cast<uint32_t>(i));
    out[i] = static_cast<uint8_t>(format == 0 ? e4m3_encode(x) : e2m1_encode(x));
  }
}

}  // namespace

cudaError_t launch_fp8_scales(const float* absmax, float* scales, int n, cudaStream_t st) {
  fp8_scales_kernel<<<(n + 255) / 256, 256, 0, st>>>(absmax, scales, n);
  return cudaGetLastError();
}

cudaError_t launch_encode_bits(int format, uint32_t first, int64_t n, uint8_t* out, int num_sms,
                               cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  encode_bits_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(format, first, n, out);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint8_t* kc,
                                     uint8_t* vc, const int32_t* slots, int T, int hkv, int d,
                                     int bs, int64_t nb, int kv_dtype, float k_scale,
                                     float v_scale, int* flags, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int64_t pb = page_bytes_of(kv_dtype, bs, hkv, d);
  const int64_t db = nvfp4_data_bytes(bs, hkv, d);
  // a programmatic dependent of the previous work on the stream, like the
  // decode kernels
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(kWriteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (kv_dtype) {
    case PD_KV_BF16:
      return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel<PD_KV_BF16>, key, value, kc, vc,
                                slots, hkv, d, bs, nb, k_scale, v_scale, pb, db, flags);
    case PD_KV_FP8_E4M3:
      return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel<PD_KV_FP8_E4M3>, key, value, kc,
                                vc, slots, hkv, d, bs, nb, k_scale, v_scale, pb, db, flags);
    default:
      return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel<PD_KV_NVFP4>, key, value, kc, vc,
                                slots, hkv, d, bs, nb, k_scale, v_scale, pb, db, flags);
  }
}

cudaError_t launch_absmax(const uint16_t* data, int64_t n, float* out, int num_sms,
                          cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 2047) / 2048;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  absmax_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(data, n, out);
  return cudaGetLastError();
}

}  // namespace pd
