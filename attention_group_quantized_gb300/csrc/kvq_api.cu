// kvq_api.cu -- the C ABI of libkvq: argument validation, cache layout,
// tensor-map encoding and dispatch to the kernels.  Nothing here synchronises
// or allocates device memory (apart from the driver's own resources for the
// graphs that replay repeated host-buffer decode steps, at most 16 per
// process); every launch goes to the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>
#include <numeric>
#include <vector>

#include "kvq_internal.h"

namespace kvq {

// (Per-device values cached in atomics: host threads may race to fill an
// entry, and they all store the same value.)
int device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

CUresult encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                              uint32_t box1, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

static bool shape_ok(const kvq_cache& c) {
  return c.B > 0 && c.Hkv > 0 && c.Hkv <= KVQ_MAX_HKV && c.Tcap > 0 && c.Tcap % KVQ_TILE_TOKENS == 0 &&
         (c.D == 64 || c.D == 128) && c.head_bits != nullptr;
}

bool resolve_layout(const kvq_cache& c, HeadLayout* out) {
  memset(out, 0, sizeof(*out));
  if (!shape_ok(c)) return false;
  const int64_t per_tok_base = static_cast<int64_t>(c.B) * c.Tcap;
  int64_t off = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const int want = pass == 0 ? 8 : 4;
    if (pass == 1) out->off4 = off;
    int idx = 0;
    for (int h = 0; h < c.Hkv; ++h) {
      const int b = c.head_bits[h];
      if (b != 4 && b != 8) return false;
      if (b != want) continue;
      out->bits[h] = static_cast<int8_t>(b);
      out->plane_idx[h] = idx++;
      out->plane_off[h] = off;
      off += per_tok_base * (c.D * b / 8);
    }
    (pass == 0 ? out->n8 : out->n4) = idx;
  }
  return true;
}

static int64_t codes_bytes(const kvq_cache& c) {
  HeadLayout hl;
  if (!resolve_layout(c, &hl)) return -1;
  return hl.off4 + static_cast<int64_t>(hl.n4) * c.B * c.Tcap * (c.D / 2);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A caller's policy (or the defaults) checked and resolved.
static bool resolve_policy(const kvq_policy* in, Policy* out) {
  *out = Policy{};
  if (in == nullptr) return true;
  // the ring depth is even: the decode's two table warps take even and odd
  // tiles, and with an even depth every slot's fills all go to one of them,
  // which then waits on each of that slot's phases in turn
  if ((in->decode_ring_tiles != 2 && in->decode_ring_tiles != 4) || in->decode_l2_warm_tiles < 0 ||
      in->decode_l2_warm_tiles > 16 || in->wait_limit_us < 1 || in->wait_limit_us > 60000000u)
    return false;
  out->ring = in->decode_ring_tiles;
  out->l2_warm = in->decode_l2_warm_tiles;
  out->wait_ns = static_cast<uint64_t>(in->wait_limit_us) * 1000u;
  out->issue_limit = in->test_issue_limit < 0 ? -1 : in->test_issue_limit;
  return true;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

int64_t kvq_cache_codes_bytes(const kvq_cache* cache) {
  if (cache == nullptr) return -1;
  return codes_bytes(*cache);
}

int64_t kvq_cache_sz_bytes(const kvq_cache* cache) {
  if (cache == nullptr || !shape_ok(*cache)) return -1;
  return static_cast<int64_t>(cache->Hkv) * cache->B * cache->Tcap * (cache->D / KVQ_GROUP) * 4;
}

int64_t kvq_cache_head_offset(const kvq_cache* cache, int32_t h) {
  if (cache == nullptr) return -1;
  HeadLayout hl;
  if (!resolve_layout(*cache, &hl) || h < 0 || h >= cache->Hkv) return -1;
  return hl.plane_off[h];
}

void kvq_policy_default(kvq_policy* policy) {
  if (policy == nullptr) return;
  const Policy d{};
  policy->decode_ring_tiles = d.ring;
  policy->decode_l2_warm_tiles = d.l2_warm;
  policy->wait_limit_us = static_cast<uint32_t>(d.wait_ns / 1000u);
  policy->test_issue_limit = d.issue_limit;
}

const char* kvq_status_str(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
    case KVQ_ERR_NONFINITE: return "non-finite input or fp16 overflow";
    case KVQ_ERR_BOUNDS: return "device index check failed (debug build)";
  }
  return "unknown status";
}

}  // extern "C"

// kvq_quantize, optionally skipping the rows at positions >= lens[b]
static kvq_status quantize_impl(const void* x, int64_t sx_b, int64_t sx_h, int64_t sx_t, int32_t t0, int32_t nt,
                                const kvq_cache* dst, const int32_t* lens, int32_t* dev_status, void* stream) {
  if (dst == nullptr || x == nullptr || dst->codes == nullptr || dst->sz == nullptr) return KVQ_ERR_INVALID_ARG;
  if (dst->D != 64 && dst->D != 128 && dst->D > 0) return KVQ_ERR_UNSUPPORTED;
  QuantizeArgs a;
  if (!resolve_layout(*dst, &a.layout)) return KVQ_ERR_INVALID_ARG;
  if (t0 < 0 || nt < 0 || static_cast<int64_t>(t0) + nt > dst->Tcap) return KVQ_ERR_INVALID_ARG;
  if (sx_b < 0 || sx_h < 0 || sx_t < 0) return KVQ_ERR_INVALID_ARG;
  // every row start must be 16-byte aligned (rows are read as 16-byte vectors)
  if (!aligned16(x) || (sx_b % 8) || (sx_h % 8) || (sx_t % 8)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(dst->codes) || !aligned16(dst->sz)) return KVQ_ERR_INVALID_ARG;
  if (nt == 0) return KVQ_OK;
  a.x = static_cast<const uint16_t*>(x);
  a.sx_b = sx_b; a.sx_h = sx_h; a.sx_t = sx_t;
  a.t0 = t0; a.nt = nt;
  a.codes = dst->codes; a.sz = dst->sz;
  a.B = dst->B; a.Hkv = dst->Hkv; a.Tcap = dst->Tcap; a.D = dst->D;
  a.status = dev_status;
  a.lens = lens;
  return launch_quantize(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" {

kvq_status kvq_quantize(const void* x, int64_t sx_b, int64_t sx_h, int64_t sx_t, int32_t t0, int32_t nt,
                        const kvq_cache* dst, int32_t* dev_status, void* stream) {
  return quantize_impl(x, sx_b, sx_h, sx_t, t0, nt, dst, nullptr, dev_status, stream);
}

size_t kvq_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D) {
  if (B <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv || (D != 64 && D != 128)) return 0;
  return decode_workspace_bytes(B, Hq, Hkv, D, decode_num_ctas(D));
}

static bool same_cache_shape(const kvq_cache& a, const kvq_cache& b) {
  if (a.B != b.B || a.Hkv != b.Hkv || a.Tcap != b.Tcap || a.D != b.D) return false;
  if (a.head_bits == nullptr || b.head_bits == nullptr) return false;
  for (int h = 0; h < a.Hkv && h < KVQ_MAX_HKV; ++h)
    if (a.head_bits[h] != b.head_bits[h]) return false;
  return true;
}

}  // extern "C"

// A block table's checks: the caches are page pools of 64-token pages.
static bool table_ok(const kvq_block_table* t, const kvq_cache& pool) {
  return t != nullptr && t->pages != nullptr && (reinterpret_cast<uintptr_t>(t->pages) & 3u) == 0 && t->B > 0 &&
         t->max_pages > 0 && pool.Tcap == KVQ_TILE_TOKENS &&
         static_cast<int64_t>(t->max_pages) * KVQ_TILE_TOKENS < (int64_t(1) << 31);
}

// Decode over contiguous caches (table == nullptr) or page pools.
static kvq_status decode_impl(const void* q, const kvq_cache* k, const kvq_cache* v, const kvq_block_table* table,
                              const int32_t* seq_lens, int32_t Hq, float softmax_scale, void* out, int32_t out_dtype,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream,
                              const kvq_policy* policy = nullptr) {
  if (q == nullptr || k == nullptr || v == nullptr || seq_lens == nullptr || out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (k->codes == nullptr || k->sz == nullptr || v->codes == nullptr || v->sz == nullptr) return KVQ_ERR_INVALID_ARG;
  if (k->D > 0 && k->D != 64 && k->D != 128) return KVQ_ERR_UNSUPPORTED;
  DecodeArgs a;
  if (!resolve_layout(*k, &a.layout) || !same_cache_shape(*k, *v)) return KVQ_ERR_INVALID_ARG;
  if (table != nullptr && !table_ok(table, *k)) return KVQ_ERR_INVALID_ARG;
  if (Hq <= 0 || Hq % k->Hkv) return KVQ_ERR_INVALID_ARG;
  if (Hq / k->Hkv > 8) return KVQ_ERR_UNSUPPORTED;
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k->codes) || !aligned16(k->sz) || !aligned16(v->codes) || !aligned16(v->sz) ||
      !aligned16(out) || (workspace != nullptr && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return KVQ_ERR_INVALID_ARG;
  // TMA row coordinates are 32-bit
  if (static_cast<int64_t>(k->Hkv) * k->B * k->Tcap >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  a.q = static_cast<const uint16_t*>(q);
  a.k = k;
  a.v = v;
  a.seq_lens = seq_lens;
  a.Hq = Hq;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.status = dev_status;
  if (!resolve_policy(policy, &a.pol)) return KVQ_ERR_INVALID_ARG;
  if (table != nullptr) {
    a.bt = table->pages;
    a.bt_B = table->B;
    a.bt_max_pages = table->max_pages;
  }
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}

extern "C" {

kvq_status kvq_decode_attention(const void* q, const kvq_cache* k, const kvq_cache* v, const int32_t* seq_lens,
                                int32_t Hq, float softmax_scale, void* out, int32_t out_dtype, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return decode_impl(q, k, v, nullptr, seq_lens, Hq, softmax_scale, out, out_dtype, workspace, workspace_bytes,
                     dev_status, stream);
}

kvq_status kvq_decode_attention_ex(const void* q, const kvq_cache* k, const kvq_cache* v, const int32_t* seq_lens,
                                   int32_t Hq, float softmax_scale, void* out, int32_t out_dtype, void* workspace,
                                   size_t workspace_bytes, const kvq_policy* policy, int32_t* dev_status,
                                   void* stream) {
  return decode_impl(q, k, v, nullptr, seq_lens, Hq, softmax_scale, out, out_dtype, workspace, workspace_bytes,
                     dev_status, stream, policy);
}

kvq_status kvq_decode_attention_paged(const void* q, const kvq_cache* k_pool, const kvq_cache* v_pool,
                                      const kvq_block_table* table, const int32_t* seq_lens, int32_t Hq,
                                      float softmax_scale, void* out, int32_t out_dtype, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (table == nullptr) return KVQ_ERR_INVALID_ARG;
  return decode_impl(q, k_pool, v_pool, table, seq_lens, Hq, softmax_scale, out, out_dtype, workspace,
                     workspace_bytes, dev_status, stream);
}

kvq_status kvq_quantize_paged(const void* x, int64_t sx_b, int64_t sx_h, int64_t sx_t, int32_t t0, int32_t nt,
                              const kvq_cache* pool, const kvq_block_table* table, int32_t* dev_status,
                              void* stream) {
  if (pool == nullptr || x == nullptr || pool->codes == nullptr || pool->sz == nullptr) return KVQ_ERR_INVALID_ARG;
  if (pool->D != 64 && pool->D != 128 && pool->D > 0) return KVQ_ERR_UNSUPPORTED;
  QuantizeArgs a;
  if (!resolve_layout(*pool, &a.layout) || !table_ok(table, *pool)) return KVQ_ERR_INVALID_ARG;
  if (t0 < 0 || nt < 0 || static_cast<int64_t>(t0) + nt > static_cast<int64_t>(table->max_pages) * KVQ_TILE_TOKENS)
    return KVQ_ERR_INVALID_ARG;
  if (sx_b < 0 || sx_h < 0 || sx_t < 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (sx_b % 8) || (sx_h % 8) || (sx_t % 8)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(pool->codes) || !aligned16(pool->sz)) return KVQ_ERR_INVALID_ARG;
  if (nt == 0) return KVQ_OK;
  a.x = static_cast<const uint16_t*>(x);
  a.sx_b = sx_b; a.sx_h = sx_h; a.sx_t = sx_t;
  a.t0 = t0; a.nt = nt;
  a.codes = pool->codes; a.sz = pool->sz;
  a.B = pool->B; a.Hkv = pool->Hkv; a.Tcap = pool->Tcap; a.D = pool->D;
  a.status = dev_status;
  a.bt = table->pages;
  a.bt_B = table->B;
  a.bt_max_pages = table->max_pages;
  return launch_quantize(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // extern "C"

// One decode step; with q_src set, the append launch also copies q_bytes
// from q_src (any device-visible memory) to q, the decode's query buffer.
static kvq_status decode_step_impl(const void* q, const void* q_src, size_t q_bytes, const void* k_new,
                                   const void* v_new, const kvq_cache* k, const kvq_cache* v,
                                   const kvq_block_table* table, const int32_t* seq_lens, int32_t Hq,
                                   float softmax_scale, void* out, int32_t out_dtype, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  // every check of the decode call first, so that nothing is appended unless both launches are valid
  if (q == nullptr || k == nullptr || v == nullptr || seq_lens == nullptr || out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (k->codes == nullptr || k->sz == nullptr || v->codes == nullptr || v->sz == nullptr) return KVQ_ERR_INVALID_ARG;
  if (k->D > 0 && k->D != 64 && k->D != 128) return KVQ_ERR_UNSUPPORTED;
  AppendArgs a;
  if (!resolve_layout(*k, &a.layout) || !same_cache_shape(*k, *v)) return KVQ_ERR_INVALID_ARG;
  if (table != nullptr && !table_ok(table, *k)) return KVQ_ERR_INVALID_ARG;
  if (Hq <= 0 || Hq % k->Hkv) return KVQ_ERR_INVALID_ARG;
  if (Hq / k->Hkv > 8) return KVQ_ERR_UNSUPPORTED;
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k->codes) || !aligned16(k->sz) || !aligned16(v->codes) || !aligned16(v->sz) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(k->Hkv) * k->B * k->Tcap >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  const int nseq = table != nullptr ? table->B : k->B;
  if (nseq > 4096) return KVQ_ERR_UNSUPPORTED;   // the decode kernel's shared memory holds up to 4096 lengths
  const size_t need = kvq_decode_workspace_bytes(nseq, Hq, k->Hkv, k->D);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return KVQ_ERR_WORKSPACE;
  if (q_src != nullptr && (!aligned16(q_src) || (q_bytes & 15u))) return KVQ_ERR_INVALID_ARG;
  a.q_src = q_src;
  a.q_dst = const_cast<void*>(q);
  a.q_bytes = q_src != nullptr ? q_bytes : 0;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_codes = k->codes; a.k_sz = k->sz;
  a.v_codes = v->codes; a.v_sz = v->sz;
  a.seq_lens = seq_lens;
  a.B = k->B; a.Hkv = k->Hkv; a.Tcap = k->Tcap; a.D = k->D;
  a.status = dev_status;
  if (table != nullptr) {
    a.bt = table->pages;
    a.bt_B = table->B;
    a.bt_max_pages = table->max_pages;
  }
  if (launch_append(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return decode_impl(q, k, v, table, seq_lens, Hq, softmax_scale, out, out_dtype, workspace, workspace_bytes,
                     dev_status, stream);
}

// ---- repeated decode steps replayed from a CUDA graph ----
// A serving loop issues the same step every token: the same buffers, caches
// and scalars, only the contents (lengths, new rows, cache codes) change, and
// the kernels read those at run time.  The second call with a given key
// captures the step's launches on an internal stream into a graph; every
// later call with that key launches the graph (one launch call, no
// tensor-map encoding).  The key holds every value the launches are built
// from: the device, each pointer and size argument, both caches' fields and
// their per-head bit widths.  At most kStepGraphs graphs are kept, for the
// life of the process; further keys run their launches directly.
namespace {

constexpr size_t kStepGraphs = 16;
constexpr size_t kStepSeen = 32;

struct StepGraph {
  std::vector<uint8_t> key;
  cudaGraphExec_t exec;
};

std::mutex g_step_mu;
std::vector<StepGraph> g_step_graphs;
std::vector<std::vector<uint8_t>> g_step_seen;   // keys met once, oldest first
cudaStream_t g_capture_stream[64] = {};

void key_put(std::vector<uint8_t>& key, const void* p, size_t n) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  key.insert(key.end(), b, b + n);
}
template <class T>
void key_val(std::vector<uint8_t>& key, T v) {
  key_put(key, &v, sizeof(v));
}
void key_cache(std::vector<uint8_t>& key, const kvq_cache* c) {
  key_val(key, c->codes);
  key_val(key, c->sz);
  key_val(key, c->head_bits);
  key_val(key, c->B);
  key_val(key, c->Hkv);
  key_val(key, c->Tcap);
  key_val(key, c->D);
  if (c->head_bits != nullptr && c->Hkv > 0 && c->Hkv <= KVQ_MAX_HKV) key_put(key, c->head_bits, c->Hkv);
}

// Runs `launch(stream)` directly, or replays it from its graph (see above).
// A stream that is itself being captured gets the launches directly.
template <class F>
kvq_status launch_or_replay(std::vector<uint8_t>& key, cudaStream_t stream, F&& launch) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  int dev = -1;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone ||
      cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return launch(stream);
  }
  key_val(key, dev);
  std::lock_guard<std::mutex> lock(g_step_mu);
  for (const StepGraph& g : g_step_graphs)
    if (g.key == key) return cudaGraphLaunch(g.exec, stream) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
  auto seen = std::find(g_step_seen.begin(), g_step_seen.end(), key);
  if (seen == g_step_seen.end() || g_step_graphs.size() >= kStepGraphs) {
    // first time (or no room): launch directly and remember the key
    if (seen == g_step_seen.end() && g_step_graphs.size() < kStepGraphs) {
      if (g_step_seen.size() >= kStepSeen) g_step_seen.erase(g_step_seen.begin());
      g_step_seen.push_back(key);
    }
    return launch(stream);
  }
  g_step_seen.erase(seen);
  if (g_capture_stream[dev] == nullptr &&
      cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
    g_capture_stream[dev] = nullptr;
    cudaGetLastError();
    return launch(stream);
  }
  cudaStream_t cap = g_capture_stream[dev];
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return launch(stream);
  }
  const kvq_status r = launch(cap);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
  cudaGraphExec_t exec = nullptr;
  const bool made = r == KVQ_OK && ec == cudaSuccess && graph != nullptr &&
                    cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
  if (graph != nullptr) cudaGraphDestroy(graph);
  if (!made) {
    cudaGetLastError();
    // a rejected argument is rejected again without launching; anything
    // else runs directly
    return r != KVQ_OK ? r : launch(stream);
  }
  g_step_graphs.push_back(StepGraph{key, exec});
  return cudaGraphLaunch(exec, stream) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_step(const void* q, const void* k_new, const void* v_new, const kvq_cache* k,
                           const kvq_cache* v, const int32_t* seq_lens, int32_t Hq, float softmax_scale, void* out,
                           int32_t out_dtype, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream) {
  return decode_step_impl(q, nullptr, 0, k_new, v_new, k, v, nullptr, seq_lens, Hq, softmax_scale, out, out_dtype,
                          workspace, workspace_bytes, dev_status, stream);
}

kvq_status kvq_decode_step_paged(const void* q, const void* k_new, const void* v_new, const kvq_cache* k_pool,
                                 const kvq_cache* v_pool, const kvq_block_table* table, const int32_t* seq_lens,
                                 int32_t Hq, float softmax_scale, void* out, int32_t out_dtype, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (table == nullptr) return KVQ_ERR_INVALID_ARG;
  return decode_step_impl(q, nullptr, 0, k_new, v_new, k_pool, v_pool, table, seq_lens, Hq, softmax_scale, out,
                          out_dtype, workspace, workspace_bytes, dev_status, stream);
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of pinned (page-locked, mapped) host memory, or null for
// pageable memory.  With unified addressing the GPU reads and writes such
// memory in place over the host link.
static void* pinned_device_view(const void* host) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
  return at.devicePointer;
}

size_t kvq_decode_step_staging_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t out_dtype) {
  if (B <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv || (D != 64 && D != 128)) return 0;
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return 0;
  const size_t q = static_cast<size_t>(B) * Hq * D * 2, kv = static_cast<size_t>(B) * Hkv * D * 2;
  const size_t o = static_cast<size_t>(B) * Hq * D * (out_dtype == KVQ_OUT_F32 ? 4 : 2);
  return round256(q) + 2 * round256(kv) + round256(o);
}

kvq_status kvq_decode_step_host(const void* q_host, const void* k_new_host, const void* v_new_host,
                                const kvq_cache* k, const kvq_cache* v, const int32_t* seq_lens, int32_t Hq,
                                float softmax_scale, void* out_host, int32_t out_dtype, void* staging,
                                size_t staging_bytes, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream) {
  if (q_host == nullptr || k_new_host == nullptr || v_new_host == nullptr || out_host == nullptr || k == nullptr ||
      staging == nullptr)
    return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_decode_step_staging_bytes(k->B, Hq, k->Hkv, k->D, out_dtype);
  if (need == 0) return KVQ_ERR_INVALID_ARG;
  if (staging_bytes < need || (reinterpret_cast<uintptr_t>(staging) & 255u)) return KVQ_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(k->B) * Hq * k->D * 2, kvb = static_cast<size_t>(k->B) * k->Hkv * k->D * 2;
  const size_t ob = static_cast<size_t>(k->B) * Hq * k->D * (out_dtype == KVQ_OUT_F32 ? 4 : 2);
  uint8_t* st = static_cast<uint8_t*>(staging);
  uint8_t* d_q = st;
  uint8_t* d_k = d_q + round256(qb);
  uint8_t* d_v = d_k + round256(kvb);
  uint8_t* d_o = d_v + round256(kvb);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Pinned host buffers: no copy calls.  The append launch reads the new
  // K/V rows in place and stages q; the decode writes the output in place.
  void* p_q = pinned_device_view(q_host);
  void* p_k = p_q ? pinned_device_view(k_new_host) : nullptr;
  void* p_v = p_k ? pinned_device_view(v_new_host) : nullptr;
  void* p_o = p_v ? pinned_device_view(out_host) : nullptr;
  if (p_o != nullptr && aligned16(p_q) && aligned16(p_k) && aligned16(p_v) && aligned16(p_o)) {
    if (v == nullptr) return KVQ_ERR_INVALID_ARG;
    std::vector<uint8_t> key;
    key.reserve(192);
    for (const void* ptr : {static_cast<const void*>(d_q), static_cast<const void*>(p_q),
                            static_cast<const void*>(p_k), static_cast<const void*>(p_v),
                            static_cast<const void*>(p_o), static_cast<const void*>(seq_lens), static_cast<const void*>(workspace),
                            static_cast<const void*>(dev_status)})
      key_val(key, ptr);
    key_val(key, qb);
    key_val(key, workspace_bytes);
    key_val(key, Hq);
    key_val(key, softmax_scale);
    key_val(key, out_dtype);
    key_cache(key, k);
    key_cache(key, v);
    return launch_or_replay(key, s, [&](cudaStream_t ls) {
      return decode_step_impl(d_q, p_q, qb, p_k, p_v, k, v, nullptr, seq_lens, Hq, softmax_scale, p_o, out_dtype,
                              workspace, workspace_bytes, dev_status, ls);
    });
  }
  // pageable memory: asynchronous copies through the staging buffer
  if (cudaMemcpyAsync(d_q, q_host, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(d_k, k_new_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(d_v, v_new_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  const kvq_status r = decode_step_impl(d_q, nullptr, 0, d_k, d_v, k, v, nullptr, seq_lens, Hq, softmax_scale, d_o,
                                        out_dtype, workspace, workspace_bytes, dev_status, stream);
  if (r != KVQ_OK) return r;
  return cudaMemcpyAsync(out_host, d_o, ob, cudaMemcpyDeviceToHost, s) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_build_tile_mask(uint8_t* mask, int32_t nT, int32_t skip_num, int32_t skip_den, uint64_t seed,
                               void* stream) {
  if (mask == nullptr || nT < 1 || nT > 16384 || skip_den < 1 || skip_num < 0 || skip_num > skip_den)
    return KVQ_ERR_INVALID_ARG;
  return launch_tile_mask(mask, nT, skip_num, skip_den, seed, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

size_t kvq_head_error_stats_workspace_bytes(int32_t H) {
  return H <= 0 ? 0 : static_cast<size_t>(H) * kHeadStatsMaxChunks * 2 * sizeof(double);
}

kvq_status kvq_head_error_stats(const void* x, int32_t B, int32_t H, int32_t T, int32_t D, const int32_t* seq_lens,
                                const float* weights, int32_t bits, double* stats, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (x == nullptr || stats == nullptr || B <= 0 || H <= 0 || H > 65535 || T <= 0) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * T >= (int64_t(1) << 31)) return KVQ_ERR_INVALID_ARG;   // rows in 32 bits
  if (bits != 4 && bits != 8) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(stats) & 7u) != 0 ||
      (weights != nullptr && (reinterpret_cast<uintptr_t>(weights) & 3u) != 0))
    return KVQ_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < kvq_head_error_stats_workspace_bytes(H) || !aligned16(workspace))
    return KVQ_ERR_WORKSPACE;
  HeadStatsArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.w = weights;
  a.lens = seq_lens;
  a.B = B; a.H = H; a.T = T; a.D = D; a.bits = bits;
  a.part = static_cast<double*>(workspace);
  a.stats = stats;
  a.status = dev_status;
  return launch_head_stats(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_allocate_head_bits(const double* k_stats, const double* v_stats, int32_t H, int32_t n_high,
                                  int32_t low_bits, int8_t* head_bits, double* score) {
  if (k_stats == nullptr || v_stats == nullptr || head_bits == nullptr || H <= 0 || n_high < 0 || n_high > H)
    return KVQ_ERR_INVALID_ARG;
  if (low_bits != 4 && low_bits != 8) return KVQ_ERR_INVALID_ARG;
  std::vector<double> sc(static_cast<size_t>(H));
  for (int32_t h = 0; h < H; ++h) {
    const double* k = k_stats + 2 * h;
    const double* v = v_stats + 2 * h;
    sc[h] = (k[1] != 0.0 ? k[0] / k[1] : 0.0) + (v[1] != 0.0 ? v[0] / v[1] : 0.0);
    if (!std::isfinite(sc[h])) return KVQ_ERR_NONFINITE;
  }
  std::vector<int32_t> order(static_cast<size_t>(H));
  std::iota(order.begin(), order.end(), 0);
  // largest score first; a stable sort keeps equal scores in head order
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return sc[a] > sc[b]; });
  for (int32_t i = 0; i < H; ++i) head_bits[order[i]] = static_cast<int8_t>(i < n_high ? 8 : low_bits);
  if (score != nullptr) std::copy(sc.begin(), sc.end(), score);
  return KVQ_OK;
}

}  // extern "C"

static kvq_status prefill_impl(const void* q, const void* k, const void* v, int32_t B, int32_t Hq, int32_t Hkv,
                               int32_t S, int32_t D, const int32_t* seq_lens, int32_t causal, float softmax_scale,
                               const uint8_t* tile_mask, int32_t tile, const kvq_cache* k_cache,
                               const kvq_cache* v_cache, void* out, int32_t out_dtype, int32_t* dev_status,
                               void* stream, const kvq_policy* policy = nullptr) {
  if (q == nullptr || k == nullptr || v == nullptr || k_cache == nullptr || v_cache == nullptr || out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || Hq % Hkv) return KVQ_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || tile != 128 || (D != 64 && D != 128) || S % 128) return KVQ_ERR_UNSUPPORTED;
  // the kernel indexes a tile mask [nT][nT] with 32-bit integers
  if (tile_mask != nullptr && static_cast<int64_t>(S / 128) * (S / 128) >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return KVQ_ERR_INVALID_ARG;
  PrefillArgs a;
  if (!resolve_policy(policy, &a.pol)) return KVQ_ERR_INVALID_ARG;
  if (!resolve_layout(*k_cache, &a.layout) || !same_cache_shape(*k_cache, *v_cache)) return KVQ_ERR_INVALID_ARG;
  if (k_cache->B != B || k_cache->Hkv != Hkv || k_cache->D != D || k_cache->Tcap < S) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(k_cache->codes) ||
      !aligned16(k_cache->sz) || !aligned16(v_cache->codes) || !aligned16(v_cache->sz))
    return KVQ_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t sx_t = D, sx_h = static_cast<int64_t>(S) * D, sx_b = sx_h * Hkv;
  kvq_status s = quantize_impl(k, sx_b, sx_h, sx_t, 0, S, k_cache, seq_lens, dev_status, stream);
  if (s != KVQ_OK) return s;
  s = quantize_impl(v, sx_b, sx_h, sx_t, 0, S, v_cache, seq_lens, dev_status, stream);
  if (s != KVQ_OK) return s;
  a.q = static_cast<const uint16_t*>(q);
  a.k = k_cache;
  a.v = v_cache;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.S = S; a.D = D;
  a.softmax_scale = softmax_scale;
  a.tile_mask = tile_mask;
  a.out = out;
  a.out_dtype = out_dtype;
  a.status = dev_status;
  a.causal = causal;
  a.lens = seq_lens;
  return launch_prefill(a, st);
}

extern "C" {

kvq_status kvq_prefill_attention(const void* q, const void* k, const void* v, int32_t B, int32_t Hq, int32_t Hkv,
                                 int32_t S, int32_t D, int32_t causal, float softmax_scale,
                                 const uint8_t* tile_mask, int32_t tile, const kvq_cache* k_cache,
                                 const kvq_cache* v_cache, void* out, int32_t out_dtype, int32_t* dev_status,
                                 void* stream) {
  return prefill_impl(q, k, v, B, Hq, Hkv, S, D, nullptr, causal, softmax_scale, tile_mask, tile, k_cache, v_cache,
                      out, out_dtype, dev_status, stream);
}

kvq_status kvq_prefill_attention_varlen(const void* q, const void* k, const void* v, int32_t B, int32_t Hq,
                                        int32_t Hkv, int32_t S, int32_t D, const int32_t* seq_lens, int32_t causal,
                                        float softmax_scale, const uint8_t* tile_mask, int32_t tile,
                                        const kvq_cache* k_cache, const kvq_cache* v_cache, void* out,
                                        int32_t out_dtype, int32_t* dev_status, void* stream) {
  if (seq_lens == nullptr) return KVQ_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, B, Hq, Hkv, S, D, seq_lens, causal, softmax_scale, tile_mask, tile, k_cache, v_cache,
                      out, out_dtype, dev_status, stream);
}

kvq_status kvq_prefill_attention_ex(const void* q, const void* k, const void* v, int32_t B, int32_t Hq, int32_t Hkv,
                                    int32_t S, int32_t D, const int32_t* seq_lens, int32_t causal,
                                    float softmax_scale, const uint8_t* tile_mask, int32_t tile,
                                    const kvq_cache* k_cache, const kvq_cache* v_cache, void* out, int32_t out_dtype,
                                    const kvq_policy* policy, int32_t* dev_status, void* stream) {
  return prefill_impl(q, k, v, B, Hq, Hkv, S, D, seq_lens, causal, softmax_scale, tile_mask, tile, k_cache, v_cache,
                      out, out_dtype, dev_status, stream, policy);
}

}  // extern "C"
