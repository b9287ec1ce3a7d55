// Decode attention with a library-owned workspace, for callers that cannot
// allocate device memory.
//
// tq_decode_attention takes its workspace (rotated queries and split-K
// partials) from the caller.  Some callers have no way to get one at the point
// where decode attention runs: a serving process that reserved the whole
// device for its own pool at start-up, so a late cudaMalloc fails; code that
// runs inside a memory-pool or allocator callback and must not re-enter the
// allocator; a plug-in hosted by an application that owns every device buffer
// and hands out inputs and outputs only; or a latency-critical loop where the
// implicit synchronisation of cudaMalloc/cudaFree is not acceptable.
// tq_decode_attention_static computes the same thing with its workspace in a
// fixed array that belongs to the library and allocates nothing.
//
// The array is a file-scope __device__ variable of kStaticWorkspaceBytes; every
// GPU that loads libtq.so keeps it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress, once per device, with that device current, on
// the first call made on that device (that first call should therefore come
// before any stream capture).  The address is kept for the life of the process:
// after cudaDeviceReset the module and the array are unloaded and the entry point
// must not be used on that device again.  All calls share the one array and it keeps the
// previous call's contents; nothing in it has to start at zero, because the
// decode kernels write every value they later read within the same call.
// Calls that overlap on the GPU (other streams, other host threads) race on it.
#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_lock;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
cudaError_t static_workspace(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" tq_status tq_decode_attention_static(const tq_context* ctx, const void* q, int q_is_fp16, int n_layers,
                                                int batch, int n_q_heads, const tq_cache_view* k_view,
                                                const tq_cache_view* v_view, int layer_begin,
                                                const int32_t* seq_lens, int max_ctx, const int32_t* block_table,
                                                int max_blocks_per_seq, float softmax_scale, float skip_threshold,
                                                float* out, tq_stream_t stream) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_decode_workspace_bytes(ctx, n_layers, batch, n_q_heads, max_ctx);
  if (need > kStaticWorkspaceBytes) return TQ_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev != ctx->device) return TQ_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (static_workspace(dev, &ws) != cudaSuccess) return TQ_ERR_CUDA;
  return tq_decode_attention(ctx, q, q_is_fp16, n_layers, batch, n_q_heads, k_view, v_view, layer_begin, seq_lens,
                             max_ctx, block_table, max_blocks_per_seq, softmax_scale, skip_threshold, ws,
                             kStaticWorkspaceBytes, out, stream);
}
