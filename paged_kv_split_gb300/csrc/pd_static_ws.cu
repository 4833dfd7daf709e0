// pd_decode_static_ws: the decode step with its split workspace in a fixed
// device array that this library owns, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code that is handed only its input and output buffers and has
// no allocator to call - for example an operator plugged into another
// framework's runtime, which owns all device memory and forbids cudaMalloc
// from inside the plugin, or a caller whose memory budget is fixed up front.
// Such a caller cannot provide the scratch that pd_decode asks for.
//
// The scratch lives in `g_static_workspace`, a file-scope __device__ array of
// PD_STATIC_WORKSPACE_BYTES. Every device that loads libpd.so reserves it for
// the life of the process. Host code may not pass the array's name to a
// kernel (in host code it is only a stand-in symbol), so the device address is
// looked up once per device with cudaGetSymbolAddress and reused.
#include <mutex>

#include "pd_common.cuh"

namespace pd {
namespace {

__device__ __align__(256) unsigned char g_static_workspace[PD_STATIC_WORKSPACE_BYTES];

constexpr int kMaxStaticDevices = 64;

struct StaticWorkspace {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
StaticWorkspace g_static[kMaxStaticDevices];

// Device address of the array on the current device. The first call on a
// device does the lookup (with that device current) and caches it.
cudaError_t static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  StaticWorkspace& w = g_static[dev];
  std::call_once(w.once, [&w]() {
    void* p = nullptr;
    w.err = cudaGetSymbolAddress(&p, g_static_workspace);
    if (w.err == cudaSuccess) w.ptr = p;
  });
  *out = w.ptr;
  return w.err;
}

}  // namespace
}  // namespace pd

extern "C" int pd_decode_static_ws(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* seq_lens,
                                   void* out, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                                   int32_t num_splits, int32_t sliding_window, int32_t kv_dtype,
                                   float k_scale, float v_scale, void* stream) {
  // pd_decode's own checks, in its order, so that both calls answer a
  // malformed request with the same status; a split count of 0 is resolved
  // the way pd_decode resolves it
  int S = 0;
  const int rc = pd::decode_checks(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs,
                                   num_q_heads, num_kv_heads, head_dim, block_size,
                                   max_blocks_per_seq, num_blocks, scale, num_splits,
                                   sliding_window, kv_dtype, k_scale, v_scale, 0, 0, &S);
  if (rc != PD_OK || num_seqs == 0) return rc;
  // The fixed array bounds the problem size: refuse anything that would not fit.
  if (pd_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, S) >
      static_cast<size_t>(PD_STATIC_WORKSPACE_BYTES))
    return PD_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (pd::static_workspace(&ws) != cudaSuccess || ws == nullptr) return PD_ERR_CUDA;
  return pd_decode(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, S,
                   sliding_window, kv_dtype, k_scale, v_scale, ws,
                   static_cast<size_t>(PD_STATIC_WORKSPACE_BYTES), stream);
}
