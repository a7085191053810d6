// kvq_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.  Some integrations run where cudaMalloc is off limits at call time:
// code inside another framework's memory pool, a plugin whose host forbids
// device allocations, or a call site that must not reach the driver's
// allocator.  For them the decode's split scratch lives in a fixed array
// compiled into the library (one per GPU that loads it, held until exit).
#include <mutex>

#include "kvq_internal.h"

namespace kvq {
namespace {

// Largest decode workspace the entry point can serve (bytes).
constexpr size_t kNoAllocBytes = size_t(4) << 20;

static __device__ __align__(256) uint8_t g_noalloc_ws[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of g_noalloc_ws on the current device, looked up once per
// device (the host-side symbol is only a stand-in and must never be passed to
// a kernel).  nullptr if the lookup fails.
void* noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess) return nullptr;
    g_noalloc_addr[dev] = p;
  }
  return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_decode_attention_noalloc(const void* q, const kvq_cache* k, const kvq_cache* v,
                                                   const int32_t* seq_lens, int32_t Hq, float softmax_scale,
                                                   void* out, int32_t out_dtype, int32_t* dev_status,
                                                   void* stream) {
  if (k == nullptr) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_decode_workspace_bytes(k->B, Hq, k->Hkv, k->D);
  if (need > kNoAllocBytes) return KVQ_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  void* ws = noalloc_scratch(dev);
  if (ws == nullptr) return KVQ_ERR_CUDA;
  // the array keeps the previous call's contents: clear the arrival counters
  if (need > 0) {
    const size_t cnt = decode_workspace_counter_bytes(k->B, k->Hkv);
    if (cudaMemsetAsync(ws, 0, cnt, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  return kvq_decode_attention(q, k, v, seq_lens, Hq, softmax_scale, out, out_dtype, ws, kNoAllocBytes,
                              dev_status, stream);
}
