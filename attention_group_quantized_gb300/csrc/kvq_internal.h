// kvq_internal.h -- launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

// Resolved per-head layout of a cache: where each head's code plane starts,
// its bit-width and its index among the planes of the same bit-width.
struct HeadLayout {
  int64_t plane_off[KVQ_MAX_HKV];   // byte offset of the head's code plane
  int32_t plane_idx[KVQ_MAX_HKV];   // index among planes of equal bit-width
  int8_t bits[KVQ_MAX_HKV];
  int32_t n8, n4;                   // number of 8-bit / 4-bit heads
  int64_t off4;                     // byte offset of the first 4-bit plane
};

bool resolve_layout(const kvq_cache& c, HeadLayout* out);

// Resolved per-call policy (kvq_policy, or its defaults).
struct Policy {
  int32_t ring = 4;               // decode: tiles in flight into shared memory (2 .. 4)
  int32_t l2_warm = 5;            // decode: tiles per CTA prefetched into L2 before the dependency wait
  uint64_t wait_ns = 2000000000ull;   // every bounded wait
  int32_t issue_limit = -1;       // test only: tiles (decode) / Q loads (prefill) issued before stopping
};

struct QuantizeArgs {
  const uint16_t* x;
  int64_t sx_b, sx_h, sx_t;
  int32_t t0, nt;
  uint8_t* codes;
  uint32_t* sz;
  int32_t B, Hkv, Tcap, D;
  int32_t* status;
  HeadLayout layout;
  // optional block table: the cache is a page pool (B = pages, Tcap = 64) and
  // x's rows are indexed by sequence bt_B x positions
  const int32_t* bt = nullptr;
  int32_t bt_B = 0, bt_max_pages = 0;
  // optional per-sequence lengths: rows at positions t0 + t >= lens[b] are
  // skipped (contiguous caches only)
  const int32_t* lens = nullptr;
};
cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream);

// The new token of every (sequence, KV head) of K and V, written at cache
// position seq_lens[b] - 1 (one launch for both caches).
struct AppendArgs {
  const void* q_src = nullptr;      // optional copy of q (q_bytes, a multiple of 16) into q_dst,
  void* q_dst = nullptr;            // done by the same launch
  size_t q_bytes = 0;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint8_t* k_codes;
  uint32_t* k_sz;
  uint8_t* v_codes;
  uint32_t* v_sz;
  const int32_t* seq_lens;
  int32_t B, Hkv, Tcap, D;
  int32_t* status;
  HeadLayout layout;                // shared by K and V
  const int32_t* bt = nullptr;      // optional block table, as in QuantizeArgs
  int32_t bt_B = 0, bt_max_pages = 0;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

struct DecodeArgs {
  const uint16_t* q;
  const kvq_cache* k;
  const kvq_cache* v;
  HeadLayout layout;                // shared by K and V
  const int32_t* seq_lens;
  int32_t Hq;
  float softmax_scale;
  void* out;
  int32_t out_dtype;
  void* ws;
  size_t ws_bytes;
  int32_t* status;
  // optional block table: the caches are page pools (B = pages, Tcap = 64)
  const int32_t* bt = nullptr;
  int32_t bt_B = 0, bt_max_pages = 0;
  Policy pol;
};
// Number of persistent split CTAs on the current device for head dim D.
int decode_num_ctas(int D);
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int D, int num_ctas);
// Leading bytes of a decode workspace that hold its arrival counters.
size_t decode_workspace_counter_bytes(int B, int Hkv);
kvq_status launch_decode(const DecodeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  const uint16_t* q;
  const kvq_cache* k;
  const kvq_cache* v;
  HeadLayout layout;
  int32_t B, Hq, Hkv, S, D;
  float softmax_scale;
  const uint8_t* tile_mask;
  void* out;
  int32_t out_dtype;
  int32_t* status;
  int32_t causal = 1;
  const int32_t* lens = nullptr;   // device [B] sequence lengths or null
  Policy pol;
};
kvq_status launch_prefill(const PrefillArgs& a, cudaStream_t stream);

cudaError_t launch_tile_mask(uint8_t* mask, int nT, int num, int den, uint64_t seed, cudaStream_t stream);

// per-KV-head quantisation-error statistics (two launches: chunk partials, fixed-order sum)
constexpr int kHeadStatsMaxChunks = 256;
struct HeadStatsArgs {
  const uint16_t* x;        // bf16 [B][H][T][D]
  const float* w;           // [B][H][T] or null
  const int32_t* lens;      // [B] or null
  int32_t B, H, T, D, bits;
  double* part;             // [H][kHeadStatsMaxChunks][2] scratch
  double* stats;            // [H][2]
  int32_t* status;
};
int head_stats_chunks(int B, int H, int T, int D);
cudaError_t launch_head_stats(const HeadStatsArgs& a, cudaStream_t stream);

// cuTensorMapEncodeTiled, resolved from the driver at first use (no link to
// libcuda, so the library loads on machines without a GPU driver).
CUresult encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                              uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

int device_sm_count();

}  // namespace kvq
