// kvq_quantize.cu -- quantise-on-write of bf16 K/V rows into the group-quantised
// cache (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.4, group of 32
// channels per the hook of §3.2).
//
// HBM-bound: every input byte is read once and every code/scale byte written
// once.  One thread quantises one group of 32 channels on its own: four
// 16-byte loads, the group's range, one IEEE division for the scale and one
// correctly rounded reciprocal, then each code from x times the reciprocal,
// rounded by a 1.5 * 2^23 addend on the FMA pipe rather than the conversion
// unit (exact division only where that product is within 2^-13 of a
// half-integer, see code_fast), and one 32-byte (INT8) or 16-byte
// (INT4) store of codes; a warp's stores cover whole contiguous rows.  The
// result is bit-identical to the specification's IEEE fp32 arithmetic.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Division of 32-bit unsigned numerators by a divisor fixed for the launch
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up multiplier of their Figure 4.1):
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
//   q = (t + ((n - t) >> 1)) >> (l - 1),  t = mulhi(m, n),   for d >= 2.
struct FastDiv {
  uint32_t d, m, l;
  static FastDiv make(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((uint64_t(1) << f.l) < d) ++f.l;
    f.m = d <= 1 ? 0u : static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << f.l) - d)) / d + 1);
    return f;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    if (d <= 1) return n;
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> 1)) >> (l - 1);
  }
};

struct QParams {
  FastDiv div_nt, div_hkv;   // row -> (b, h, t): row = (b * Hkv + h) * nt + t
  // optional block table: the cache is a pool of B pages of Tcap = 64 tokens
  // and sequence b's token t sits in page bt[b * bt_stride + t / 64]
  const int32_t* bt;
  int32_t bt_stride;
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

// 1.5 * 2^23: adding it to a float of magnitude below 2^22 rounds that value
// to the nearest integer (ties to even) -- floats in [2^23, 2^24) are spaced
// 1 apart -- and leaves the integer in the low mantissa bits.
constexpr float kRoundAdd = 12582912.0f;
constexpr int kRoundAddBits = 0x4B400000;

// code = clamp(rne(fl(x / s)) + z, 0, qmax) on the fast path, with
// C = z + 1.5 * 2^23 (z an integer, exact):
//   t = fl(x * fl(1/s)) is within 2^-14 of x / s (two roundings of relative
//   size 2^-24 at magnitudes below 2^9) and fl(x / s) within 2^-16 of it;
//   m = fl(t + C) = C + rne(t + z), the code before clamping in m's low bits;
//   e = (m - C) - t, exactly the rounding error of t + z.
// When |e| is more than 2^-13 below 1/2, t + z and fl(x / s) + z lie on the
// same side of every half-integer, so rne(t + z) = rne(fl(x / s)) + z.
// Otherwise (and for a NaN quotient) `near` is set and the caller redoes the
// group with the exact division.
__device__ __forceinline__ int code_fast(float x, float rcp, float C, int qmax, bool& near) {
  const float t = __fmul_rn(x, rcp);
  const float m = __fadd_rn(t, C);
  const float e = __fsub_rn(__fsub_rn(m, C), t);
  near |= !(fabsf(e) <= 0.5f - 0x1p-13f);
  return min(max(__float_as_int(m) - kRoundAddBits, 0), qmax);
}

// Value i (0..31) of a group held as 16 words of raw bf16 pairs.
__device__ __forceinline__ float group_value(const uint32_t (&w)[16], int i) {
  return bf16_bits_to_float((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
}

// Codes of a group packed for the store: 8-bit, four codes per word (8
// words); 4-bit, eight codes per word (4 words).  code(i) gives value i's code.
template <class F>
__device__ __forceinline__ void pack_codes(uint32_t (&packed)[8], int bits, F code) {
#pragma unroll
  for (int k = 0; k < 8; ++k) packed[k] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t c = static_cast<uint32_t>(code(i));
    if (bits == 8) packed[i >> 2] |= c << (8 * (i & 3));
    else packed[i >> 3] |= c << (4 * (i & 7));
  }
}

// Quantise one group of 32 channels (this thread alone): w holds the 32 bf16
// values as loaded by load_group (64 bytes, 16-byte aligned source), the
// codes go to cdst (32 bytes for 8-bit, 16 for 4-bit) and the fp16
// (scale, zero) word to *szw.  The values stay packed as loaded and are
// widened where used, which keeps the thread's registers few.  Non-finite input:
// an infinity makes the range, hence the scale, infinite; a NaN is dropped by
// the min/max but gives a NaN quotient (seen on the exact path) or, in an
// otherwise all-zero group, is tested directly.
__device__ __forceinline__ void load_group(uint32_t (&w)[16], const uint16_t* src) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 raw = reinterpret_cast<const uint4*>(src)[v];
    w[4 * v] = raw.x; w[4 * v + 1] = raw.y; w[4 * v + 2] = raw.z; w[4 * v + 3] = raw.w;
  }
}

__device__ __forceinline__ void quantize_group(const uint32_t (&w)[16], int bits, uint8_t* cdst, uint32_t* szw,
                                               int32_t* status) {
  // min and max over the 32 values in bf16 pairs (exact), then the two lanes
  __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&w[0]), mx2 = mn2;
#pragma unroll
  for (int k = 1; k < 16; ++k) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
    mn2 = __hmin2(mn2, v);
    mx2 = __hmax2(mx2, v);
  }
  const float mn = fminf(__low2float(mn2), __high2float(mn2));
  const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
  const int qmax = (1 << bits) - 1;
  const float qf = static_cast<float>(qmax);
  const float lo = fminf(0.0f, mn);
  const float hi = fmaxf(0.0f, mx);
  const float range = __fsub_rn(hi, lo);

  __half scale_h = __ushort_as_half(0x3C00);  // 1.0
  int zero = 0;
  uint32_t packed[8];
  bool bad = false;
  if (range == 0.0f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float x = group_value(w, i);
      bad |= x != x;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) packed[k] = 0u;
  } else {
    scale_h = __float2half_ru(__fdiv_rn(range, qf));
    const float sf = __half2float(scale_h);
    bad = !isfinite(sf);
    const float rcp = __frcp_rn(sf);
    // zero point: one exact quotient per group
    const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.0f), qf);
    zero = static_cast<int>(zf);
    const float C = zf + kRoundAdd;   // exact
    bool near = false;
    pack_codes(packed, bits, [&](int i) { return code_fast(group_value(w, i), rcp, C, qmax, near); });
    if (near) {   // rare: some quotient is within 2^-13 of a half-integer (or NaN): exact division
      pack_codes(packed, bits, [&](int i) {
        const float q = __fdiv_rn(group_value(w, i), sf);
        bad |= q != q;
        return static_cast<int>(fminf(fmaxf(rintf(q) + zf, 0.0f), qf));
      });
    }
  }
  if (bad) report(status, KVQ_ERR_NONFINITE);
  uint4* dst = reinterpret_cast<uint4*>(cdst);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (bits == 8) dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  *szw = __half_as_ushort(scale_h) | (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(zero))) << 16);
}

// resident blocks of 256 threads per SM the register budget is sized for (tunable at build time)
#ifndef KVQ_QUANT_MIN_BLOCKS
#define KVQ_QUANT_MIN_BLOCKS 5
#endif

// One thread per (row, group): row = (b * Hkv + h) * nt + t.  (A persistent
// loop that issued the next group's loads before this group's arithmetic
// measured slower: the extra registers cost more occupancy than it gained.)
// PAGED: the cache is a page pool addressed through p.bt (a separate
// instantiation, so the contiguous kernel carries none of it).
template <int D, bool PAGED>
__global__ void __launch_bounds__(256, KVQ_QUANT_MIN_BLOCKS) quantize_kernel(const __grid_constant__ QParams p) {
  constexpr int G = D / 32;
  const int64_t n = p.rows * G;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t r = static_cast<uint32_t>(i / G);
    const int g = static_cast<int>(i % G);
    const uint32_t bh = p.div_nt.div(r);
    const int t = static_cast<int>(r - bh * p.div_nt.d);
    const uint32_t bq = p.div_hkv.div(bh);
    const int h = static_cast<int>(bh - bq * p.div_hkv.d);
    const int b = static_cast<int>(bq);
    const int bits = p.bits[h];
    int64_t pos = static_cast<int64_t>(b) * p.Tcap + p.t0 + t;
    if constexpr (PAGED) {
      const int tl = p.t0 + t;
      const int page = p.bt[static_cast<int64_t>(b) * p.bt_stride + tl / 64];
      if (page < 0 || page >= p.B) {   // a page outside the pool: report, write nothing
        if (g == 0) report(p.status, KVQ_ERR_INVALID_ARG);
        continue;
      }
      pos = static_cast<int64_t>(page) * 64 + tl % 64;
    }
    uint32_t w[16];
    load_group(w, p.x + b * p.sx_b + h * p.sx_h + t * p.sx_t + g * 32);
    quantize_group(w, bits, p.codes + p.plane_off[h] + pos * (D * bits / 8) + g * (32 * bits / 8),
                   p.sz + (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G + g, p.status);
  }
}

// Append: the new token of every (sequence b, KV head h) of K and of V, rows
// [k rows | v rows] of [b][h], written at cache position seq_lens[b] - 1.
struct AParams {
  const int32_t* bt;        // optional block table (the caches are page pools), as in QParams
  int32_t bt_stride;
  const uint4* q_src;       // optional: q vectors to stage for the decode (host memory read in place)
  uint4* q_dst;
  int64_t q_vec;            // 16-byte vectors to copy
  const uint16_t* x[2];     // k_new, v_new: bf16 [B][Hkv][D]
  uint8_t* codes[2];
  uint32_t* sz[2];
  const int32_t* seq_lens;
  int32_t* status;
  int32_t B, Hkv, Tcap;     // storage: B sequences (or pages) of Tcap tokens
  int32_t nseq, cap;        // sequences and their capacity in tokens
  int64_t plane_off[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AParams p) {
  constexpr int G = D / 32;
  // the decode launched after this kernel may begin its prologue now; it
  // waits for this grid's completion before reading memory
  grid_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.q_vec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p.q_dst[i] = p.q_src[i];
  const int64_t bhn = static_cast<int64_t>(p.nseq) * p.Hkv;
  const int64_t n = 2 * bhn * G;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / G;                 // [k rows | v rows] of [b][h]
    const int g = static_cast<int>(i % G);
    const int job = static_cast<int>(r / bhn);
    const int64_t bh = r % bhn;
    const int h = static_cast<int>(bh % p.Hkv);
    const int b = static_cast<int>(bh / p.Hkv);
    const int len = p.seq_lens[b];
    if (len < 1 || len > p.cap) {
      if (job == 0 && h == 0 && g == 0) report(p.status, KVQ_ERR_INVALID_ARG);
      continue;
    }
    const int bits = p.bits[h];
    int64_t pos = static_cast<int64_t>(b) * p.Tcap + len - 1;
    if constexpr (PAGED) {
      const int page = p.bt[static_cast<int64_t>(b) * p.bt_stride + (len - 1) / 64];
      if (page < 0 || page >= p.B) {
        if (job == 0 && h == 0 && g == 0) report(p.status, KVQ_ERR_INVALID_ARG);
        continue;
      }
      pos = static_cast<int64_t>(page) * 64 + (len - 1) % 64;
    }
    uint32_t w[16];
    load_group(w, p.x[job] + bh * D + g * 32);
    quantize_group(w, bits, p.codes[job] + p.plane_off[h] + pos * (D * bits / 8) + g * (32 * bits / 8),
                   p.sz[job] + (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G + g, p.status);
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream) {
  QParams p;
  p.x = a.x;
  p.sx_b = a.sx_b; p.sx_h = a.sx_h; p.sx_t = a.sx_t;
  p.codes = a.codes; p.sz = a.sz; p.status = a.status;
  p.B = a.B; p.Hkv = a.Hkv; p.Tcap = a.Tcap; p.t0 = a.t0; p.nt = a.nt;
  p.bt = a.bt;
  p.bt_stride = a.bt_max_pages;
  p.rows = static_cast<int64_t>(a.bt != nullptr ? a.bt_B : a.B) * a.Hkv * a.nt;
  if (p.rows >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // rows are indexed in 32 bits
  p.div_nt = FastDiv::make(static_cast<uint32_t>(a.nt));
  p.div_hkv = FastDiv::make(static_cast<uint32_t>(a.Hkv));
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane_off[h] = a.layout.plane_off[h];
    p.bits[h] = a.layout.bits[h];
  }
  if (p.rows == 0) return cudaSuccess;
  int64_t blocks = (p.rows * (a.D / 32) + 255) / 256;   // one thread per (row, group)
  const int64_t cap = int64_t(1) << 30;                   // grid-stride beyond that
  if (blocks > cap) blocks = cap;
  const unsigned g = static_cast<unsigned>(blocks);
  if (a.D == 128) {
    if (p.bt != nullptr) quantize_kernel<128, true><<<g, 256, 0, stream>>>(p);
    else quantize_kernel<128, false><<<g, 256, 0, stream>>>(p);
  } else {
    if (p.bt != nullptr) quantize_kernel<64, true><<<g, 256, 0, stream>>>(p);
    else quantize_kernel<64, false><<<g, 256, 0, stream>>>(p);
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
  p.bt = a.bt;
  p.bt_stride = a.bt_max_pages;
  p.nseq = a.bt != nullptr ? a.bt_B : a.B;
  p.cap = a.bt != nullptr ? a.bt_max_pages * 64 : a.Tcap;
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane_off[h] = a.layout.plane_off[h];
    p.bits[h] = a.layout.bits[h];
  }
  const int64_t rows = 2 * static_cast<int64_t>(p.nseq) * a.Hkv;
  int64_t blocks = (rows * (a.D / 32) + 255) / 256;   // one thread per (row, group)
  const int64_t qblocks = (p.q_vec + 255) / 256;   // one 16-byte vector per thread
  if (qblocks > blocks) blocks = qblocks;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  const unsigned g = static_cast<unsigned>(blocks);
  if (a.D == 128) {
    if (p.bt != nullptr) append_kernel<128, true><<<g, 256, 0, stream>>>(p);
    else append_kernel<128, false><<<g, 256, 0, stream>>>(p);
  } else {
    if (p.bt != nullptr) append_kernel<64, true><<<g, 256, 0, stream>>>(p);
    else append_kernel<64, false><<<g, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvq
