// kvq_quantize.cu -- quantise-on-write of bf16 K/V rows into the group-quantised
// cache (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.4, group of 32
// channels per the hook of §3.2).
//
// HBM-bound: every input byte is read once and every code/scale byte written
// once.  Each thread takes 8 consecutive channels (one 16-byte load), four
// threads form a group of 32 and agree on its range with two shuffles; codes
// are written as 8 bytes (INT8) or 4 bytes (INT4) per thread, so a warp
// stores whole contiguous rows.  All arithmetic is IEEE fp32 with explicit
// rounding intrinsics so the result is bit-identical to the specification.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

struct QParams {
  const uint16_t* x;
  int64_t sx_b, sx_h, sx_t;
  uint8_t* codes;
  uint32_t* sz;
  int32_t* status;
  int32_t B, Hkv, Tcap, t0, nt;
  int64_t rows;
  int64_t plane_off[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Quantise one row of D channels: this thread holds channels 8*sub .. 8*sub+7
// (x8, raw bf16), the four threads of a group exchange their range by
// shuffles (all 32 lanes take part; `store` false skips the writes), and the
// codes and the group's scale/zero word go to `crow` / `szrow`.
template <int D>
__device__ __forceinline__ void quantize_row(const uint4 raw, int sub, int bits, bool store, uint8_t* crow,
                                             uint32_t* szrow, int32_t* status) {
  float x[8];
  x[0] = bf16_bits_to_float(raw.x & 0xFFFFu); x[1] = bf16_bits_to_float(raw.x >> 16);
  x[2] = bf16_bits_to_float(raw.y & 0xFFFFu); x[3] = bf16_bits_to_float(raw.y >> 16);
  x[4] = bf16_bits_to_float(raw.z & 0xFFFFu); x[5] = bf16_bits_to_float(raw.z >> 16);
  x[6] = bf16_bits_to_float(raw.w & 0xFFFFu); x[7] = bf16_bits_to_float(raw.w >> 16);

  bool finite = true;
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    finite &= isfinite(x[i]);
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
  // the four threads of a group share its range
  mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));

  const int qmax = (1 << bits) - 1;
  const float lo = fminf(0.0f, mn);
  const float hi = fmaxf(0.0f, mx);
  const float range = __fsub_rn(hi, lo);

  __half scale_h = __ushort_as_half(0x3C00);  // 1.0
  int zero = 0;
  int code[8];
  if (range == 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) code[i] = 0;
  } else {
    scale_h = __float2half_ru(__fdiv_rn(range, static_cast<float>(qmax)));
    const float sf = __half2float(scale_h);
    finite &= isfinite(sf);
    zero = min(max(__float2int_rn(__fdiv_rn(-lo, sf)), 0), qmax);
#pragma unroll
    for (int i = 0; i < 8; ++i) code[i] = min(max(__float2int_rn(__fdiv_rn(x[i], sf)) + zero, 0), qmax);
  }
  if (!store) return;
  if (!finite) report(status, KVQ_ERR_NONFINITE);

  if (bits == 8) {
    uint2 w;
    w.x = code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24);
    w.y = code[4] | (code[5] << 8) | (code[6] << 16) | (code[7] << 24);
    *reinterpret_cast<uint2*>(crow + sub * 8) = w;
  } else {
    const uint32_t w = code[0] | (code[1] << 4) | (code[2] << 8) | (code[3] << 12) | (code[4] << 16) |
                       (code[5] << 20) | (code[6] << 24) | (code[7] << 28);
    *reinterpret_cast<uint32_t*>(crow + sub * 4) = w;
  }
  if ((sub & 3) == 0) {
    const uint32_t zh = __half_as_ushort(__int2half_rn(zero));
    szrow[sub / 4] = __half_as_ushort(scale_h) | (zh << 16);
  }
}

template <int D>
__global__ void __launch_bounds__(256) quantize_kernel(const __grid_constant__ QParams p) {
  constexpr int TPR = D / 8;        // threads per row
  constexpr int RPW = 32 / TPR;     // rows per warp
  constexpr int G = D / 32;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t base = warp * RPW; base < p.rows; base += nwarps * RPW) {
    const int64_t row = base + lane / TPR;
    const bool live = row < p.rows;
    const int64_t r = live ? row : base;  // dead lanes shadow a live row (no stores)
    const int t = static_cast<int>(r % p.nt);
    const int64_t bh = r / p.nt;
    const int h = static_cast<int>(bh % p.Hkv);
    const int b = static_cast<int>(bh / p.Hkv);

    const uint4 raw = *reinterpret_cast<const uint4*>(p.x + b * p.sx_b + h * p.sx_h + t * p.sx_t + sub * 8);
    const int bits = p.bits[h];
    const int64_t pos = static_cast<int64_t>(b) * p.Tcap + p.t0 + t;
    quantize_row<D>(raw, sub, bits, live, p.codes + p.plane_off[h] + pos * (D * bits / 8),
                    p.sz + (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G, p.status);
  }
}

// Append: the new token of every (sequence b, KV head h) of K and of V, rows
// [k rows | v rows] of [b][h], written at cache position seq_lens[b] - 1.
struct AParams {
  const uint4* q_src;       // optional: q vectors to stage for the decode (host memory read in place)
  uint4* q_dst;
  int64_t q_vec;            // 16-byte vectors to copy
  const uint16_t* x[2];     // k_new, v_new: bf16 [B][Hkv][D]
  uint8_t* codes[2];
  uint32_t* sz[2];
  const int32_t* seq_lens;
  int32_t* status;
  int32_t B, Hkv, Tcap;
  int64_t plane_off[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

template <int D>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AParams p) {
  constexpr int TPR = D / 8;
  constexpr int RPW = 32 / TPR;
  constexpr int G = D / 32;
  // the decode launched after this kernel may begin its prologue now; it
  // waits for this grid's completion before reading memory
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.q_vec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p.q_dst[i] = p.q_src[i];
  const int64_t rows = 2 * static_cast<int64_t>(p.B) * p.Hkv;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp * RPW; base < rows; base += nwarps * RPW) {
    const int64_t row = base + lane / TPR;
    const bool live = row < rows;
    const int64_t r = live ? row : base;
    const int job = static_cast<int>(r / (static_cast<int64_t>(p.B) * p.Hkv));
    const int64_t bh = r % (static_cast<int64_t>(p.B) * p.Hkv);
    const int h = static_cast<int>(bh % p.Hkv);
    const int b = static_cast<int>(bh / p.Hkv);
    const int len = p.seq_lens[b];
    const bool in_range = len >= 1 && len <= p.Tcap;
    if (live && !in_range && sub == 0 && job == 0 && h == 0) report(p.status, KVQ_ERR_INVALID_ARG);
    const uint4 raw = *reinterpret_cast<const uint4*>(p.x[job] + bh * D + sub * 8);
    const int bits = p.bits[h];
    const int64_t pos = static_cast<int64_t>(b) * p.Tcap + (in_range ? len - 1 : 0);
    quantize_row<D>(raw, sub, bits, live && in_range, p.codes[job] + p.plane_off[h] + pos * (D * bits / 8),
                    p.sz[job] + (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G, p.status);
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream) {
  QParams p;
  p.x = a.x;
  p.sx_b = a.sx_b; p.sx_h = a.sx_h; p.sx_t = a.sx_t;
  p.codes = a.codes; p.sz = a.sz; p.status = a.status;
  p.B = a.B; p.Hkv = a.Hkv; p.Tcap = a.Tcap; p.t0 = a.t0; p.nt = a.nt;
  p.rows = static_cast<int64_t>(a.B) * a.Hkv * a.nt;
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane_off[h] = a.layout.plane_off[h];
    p.bits[h] = a.layout.bits[h];
  }
  if (p.rows == 0) return cudaSuccess;
  const int rows_per_block = 256 / (a.D / 8) * 1;  // threads / threads-per-row
  int64_t blocks = (p.rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (a.D == 128) {
    quantize_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  } else {
    quantize_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  AParams p;
  p.q_src = static_cast<const uint4*>(a.q_src);
  p.q_dst = static_cast<uint4*>(a.q_dst);
  p.q_vec = a.q_src != nullptr ? static_cast<int64_t>(a.q_bytes / 16) : 0;
  p.x[0] = a.k_new; p.x[1] = a.v_new;
  p.codes[0] = a.k_codes; p.codes[1] = a.v_codes;
  p.sz[0] = a.k_sz; p.sz[1] = a.v_sz;
  p.seq_lens = a.seq_lens;
  p.status = a.status;
  p.B = a.B; p.Hkv = a.Hkv; p.Tcap = a.Tcap;
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane_off[h] = a.layout.plane_off[h];
    p.bits[h] = a.layout.bits[h];
  }
  const int64_t rows = 2 * static_cast<int64_t>(a.B) * a.Hkv;
  const int rows_per_block = 256 / (a.D / 8);
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t qblocks = (p.q_vec + 255) / 256;   // one 16-byte vector per thread
  if (qblocks > blocks) blocks = qblocks;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (a.D == 128) {
    append_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  } else {
    append_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvq
