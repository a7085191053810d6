// kvq_quantize.cu -- quantise-on-write of bf16 K/V rows into the group-quantised
// cache (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.4, group of 32
// channels per the hook of §3.2), and per-head quantisation-error statistics
// for the per-head bit allocation of the same section.
//
// HBM-bound: every input byte is read once and every code/scale byte written
// once.  One thread quantises one group of 32 channels on its own: four
// 16-byte loads, the group's range, one IEEE division for the scale, then
// each code from x times an approximate reciprocal of the scale, rounded by a
// 1.5 * 2^23 addend inside the same FMA, two values per instruction (paired
// fp32).  The exact remainder x - u * s tells whether that rounding is the
// specification's (see rne_div); the rare quarter-groups where it might not
// be are redone value by value.  One 32-byte (INT8) or 16-byte (INT4) store
// of codes per group; a warp's stores cover whole contiguous rows.  The result
// is bit-identical to the specification's IEEE fp32 arithmetic.
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
  const int32_t* lens;      // optional per-sequence lengths (contiguous caches only)
  const uint16_t* x;
  int64_t sx_b, sx_h, sx_t;
  uint8_t* codes;
  uint32_t* sz;
  int32_t* status;
  int32_t B, Hkv, Tcap, t0, nt;
  int64_t rows;
  int64_t codes_bytes;      // size of the code buffer (the debug build's index checks)
  int64_t plane_off[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

// Debug build: a group's codes (nbytes from byte offset off) and its
// scale/zero word (index si) inside their buffers.
__device__ __forceinline__ bool group_dst_ok(int64_t off, int nbytes, int64_t si, int64_t codes_bytes,
                                             int64_t sz_words, int32_t* status) {
  return KVQ_IN_RANGE(off >= 0 && off + nbytes <= codes_bytes && si >= 0 && si < sz_words, status);
}

// 1.5 * 2^23: adding it to a float of magnitude below 2^22 rounds that value
// to the nearest integer (ties to even) -- floats in [2^23, 2^24) are spaced
// 1 apart -- and leaves the integer in the low mantissa bits (its bit pattern
// 0x4B400000 has a zero low byte).
constexpr float kRoundAdd = 12582912.0f;

// max(a, b, c), NaN if any input is NaN (three-input form, sm_100 and later)
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// rne(a / s), ties to even, for a bf16 value a and an fp16 scale s with
// |a / s| <= 256, given any r within 2^-21 (relative) of 1/s:
//   u = rne(a * r) is at most one step from rne(a / s);
//   d = a - u * s is exact in fp32 (u * s has at most 20 significant bits and
//     |d| <= 1.5 s while s >= |a| / 256, so d fits in 24 bits);
//   u moves one step towards a / s when |d| > s / 2, or when |d| = s / 2
//     (a / s is a half-integer) and u is odd.
// For such a and s this is also rne(fl(a / s)), the IEEE fp32 quotient
// rounded: fl(a / s) equals a half-integer h only when a / s does (a nonzero
// a - h * s is a multiple of 2^(e_a - 20), while fl(a / s) = h needs
// |a - h * s| < s * ulp(h) / 2, about 2^(e_a - 23)), and otherwise stays on
// the same side of every half-integer as a / s.  (Checked against the IEEE
// quotient for every finite bf16 a and fp16 scales from 2^-24 to 2^8.)
__device__ __forceinline__ float rne_div(float a, float s, float r) {
  float u = __fsub_rn(__fmaf_rn(a, r, kRoundAdd), kRoundAdd);
  const float d = __fmaf_rn(-u, s, a);
  const float ad = fabsf(d), hs = 0.5f * s;
  if (ad > hs || (ad == hs && (static_cast<int>(u) & 1) != 0)) u = __fadd_rn(u, copysignf(1.0f, d));
  return u;
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Load one group of 32 bf16 values (64 bytes, 16-byte aligned source) as 16
// words of raw bf16 pairs; they stay packed and are widened where used.
__device__ __forceinline__ void load_group(uint32_t (&w)[16], const uint16_t* src) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 raw = reinterpret_cast<const uint4*>(src)[v];
    w[4 * v] = raw.x; w[4 * v + 1] = raw.y; w[4 * v + 2] = raw.z; w[4 * v + 3] = raw.w;
  }
}

// A group's parameters: the range widened to contain 0, the fp16 scale
// s = round-up(range / qmax) (one IEEE division), the zero point
// z = clamp(rne(-lo / s), 0, qmax) (rne_div), and the fast path's constants.
// Non-finite input: an infinity makes the range, hence the scale, infinite; a
// NaN is dropped by the min/max but shows in the fast path's largest remainder
// (or, in an otherwise all-zero group, in group_has_nan).
struct GroupParams {
  __half scale_h;   // 1 when the range is 0
  float mn, mx;     // the group's min and max (before widening)
  float sf, rcp, zf, C;   // scale, approximate 1/scale, zero point, zero + 1.5 * 2^23
  int qmax;
  bool flat;        // range 0 (all zeros, or NaN among zeros): every code 0
  bool bad;         // non-finite scale
};

__device__ __forceinline__ GroupParams group_params(const uint32_t (&w)[16], int bits) {
  // min and max over the 32 values in bf16 pairs (exact), then the two lanes
  __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&w[0]), mx2 = mn2;
#pragma unroll
  for (int k = 1; k < 16; ++k) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
    mn2 = __hmin2(mn2, v);
    mx2 = __hmax2(mx2, v);
  }
  GroupParams g;
  g.mn = fminf(__low2float(mn2), __high2float(mn2));
  g.mx = fmaxf(__low2float(mx2), __high2float(mx2));
  g.qmax = (1 << bits) - 1;
  const float qf = static_cast<float>(g.qmax);
  const float lo = fminf(0.0f, g.mn);
  const float hi = fmaxf(0.0f, g.mx);
  const float range = __fsub_rn(hi, lo);
  g.flat = range == 0.0f;
  g.scale_h = __ushort_as_half(0x3C00);  // 1.0
  g.sf = 1.0f; g.rcp = 1.0f; g.zf = 0.0f; g.C = kRoundAdd;
  g.bad = false;
  if (!g.flat) {
    g.scale_h = __float2half_ru(__fdiv_rn(range, qf));
    g.sf = __half2float(g.scale_h);
    g.bad = !isfinite(g.sf);
    g.rcp = rcp_approx(g.sf);
    g.zf = fminf(fmaxf(rne_div(-lo, g.sf, g.rcp), 0.0f), qf);
    g.C = g.zf + kRoundAdd;   // exact
  }
  return g;
}

// Whether some code of the group is clamped: rne(mx / s) + z > qmax or
// rne(mn / s) + z < 0, decided exactly from the remainders against the
// half-integers k + 1/2 (k = qmax - z) and -z - 1/2 (exact as in rne_div), a
// remainder of 0 being a tie that rounds to the even side.  Codes are
// monotone in x, so no other value is clamped when these two are not.
__device__ __forceinline__ bool group_clamps(const GroupParams& g) {
  const float k = static_cast<float>(g.qmax) - g.zf;
  const float rt = __fmaf_rn(-(k + 0.5f), g.sf, g.mx);
  const float rb = __fmaf_rn(g.zf + 0.5f, g.sf, g.mn);
  return rt > 0.0f || (rt == 0.0f && (static_cast<int>(k) & 1) != 0) ||
         rb < 0.0f || (rb == 0.0f && (static_cast<int>(g.zf) & 1) != 0);
}

// The specification's code of one value (a NaN gives code 0, as the
// specification's clamp of a NaN quotient does).
__device__ __forceinline__ int code_exact(float x, const GroupParams& g) {
  return static_cast<int>(fminf(fmaxf(__fadd_rn(rne_div(x, g.sf, g.rcp), g.zf), 0.0f), static_cast<float>(g.qmax)));
}

__device__ __forceinline__ bool group_has_nan(const uint32_t (&w)[16]) {
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float2 x2 = bf16x2_to_float2(w[k]);
    bad |= (x2.x != x2.x) || (x2.y != x2.y);
  }
  return bad;
}

// Quarter v (values 8v .. 8v+7) of a group re-read from `src` (an L1 hit),
// passed to f(j, x) with j = 0..7.  Used by the rare paths, which run a
// quarter at a time in a rolled loop so the group's registers are not all
// live at once.
template <class F>
__device__ __forceinline__ void quarter_values(const uint16_t* src, int v, F f) {
  const uint4 raw = reinterpret_cast<const uint4*>(src)[v];
  const uint32_t q4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) f(j, bf16_bits_to_float((j & 1) ? (q4[j >> 1] >> 16) : (q4[j >> 1] & 0xFFFFu)));
}

// Quantise one group of 32 channels (this thread alone): w holds the 32 bf16
// values as loaded by load_group from src; the codes go to cdst (32 bytes for
// 8-bit, 16 for 4-bit) and the fp16 (scale, zero) word to *szw.
// Fast path, per pair of values: m = fl(x * r + C) holds rne(x * r) + z in its
// low mantissa bits (C's low byte is zero, so a code 0 .. qmax is m's low byte
// or nibble, gathered by byte permutes), u = m - C = rne(x * r), d = x - u * s
// exact; the code is the specification's wherever |d| < s / 2 (then u is the
// integer nearest x / s) and no code is clamped (group_clamps).  A quarter
// with some |d| at least s / 2 (a tie, or u one step off) or a NaN (the
// quarter's largest |d| is then NaN), or a clamped group, is redone with
// code_exact and stored 8 codes at a time.
__device__ __forceinline__ void quantize_group(const uint32_t (&w)[16], const uint16_t* src, int bits,
                                               uint8_t* cdst, uint32_t* szw, int32_t* status) {
  const GroupParams gp = group_params(w, bits);
  bool bad = gp.bad;
  uint32_t packed[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) packed[k] = 0u;
  unsigned redo = 0;   // quarters to redo, one bit each
  if (gp.flat) {
    bad |= group_has_nan(w);
  } else {
    const float2 r2 = make_float2(gp.rcp, gp.rcp), c2 = make_float2(gp.C, gp.C);
    const float2 nc2 = make_float2(-gp.C, -gp.C), ns2 = make_float2(-gp.sf, -gp.sf);
    const float hs = 0.5f * gp.sf;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      // the largest |d| of the quarter; a NaN anywhere makes it NaN
      float dmax = 0.0f;
      uint32_t mb[8];   // bits of m: C = z + 1.5 * 2^23 has a zero low byte, so the code is in the low bits
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float2 x2 = bf16x2_to_float2(w[4 * v + kk]);
        const float2 m2 = __ffma2_rn(x2, r2, c2);
        const float2 d2 = __ffma2_rn(__fadd2_rn(m2, nc2), ns2, x2);
        dmax = fmax3_nan(dmax, fabsf(d2.x), fabsf(d2.y));
        mb[2 * kk] = __float_as_uint(m2.x);
        mb[2 * kk + 1] = __float_as_uint(m2.y);
      }
      if (bits == 8) {   // low bytes of four m's per word
        packed[2 * v] = prmt(prmt(mb[0], mb[1], 0x0040u), prmt(mb[2], mb[3], 0x0040u), 0x5410u);
        packed[2 * v + 1] = prmt(prmt(mb[4], mb[5], 0x0040u), prmt(mb[6], mb[7], 0x0040u), 0x5410u);
      } else {           // low nibbles of eight m's, the first in bits 0-3
        uint32_t b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = (mb[2 * j] & 0x0Fu) | ((mb[2 * j + 1] << 4) & 0xF0u);
        packed[v] = prmt(prmt(b[0], b[1], 0x0040u), prmt(b[2], b[3], 0x0040u), 0x5410u);
      }
      redo |= (dmax < hs ? 0u : 1u) << v;   // false for a NaN
    }
    if (group_clamps(gp)) redo = 0xFu;
  }
  if (redo == 0u) {
    uint4* dst = reinterpret_cast<uint4*>(cdst);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (bits == 8) dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  } else {   // rare: whole group stored quarter by quarter, the flagged quarters recomputed
#pragma unroll 1
    for (int v = 0; v < 4; ++v) {
      uint32_t c8[2];
      if ((redo >> v) & 1u) {
        c8[0] = 0u;
        c8[1] = 0u;
        quarter_values(src, v, [&](int j, float x) {
          bad |= x != x;
          const uint32_t c = static_cast<uint32_t>(code_exact(x, gp));
          if (bits == 8) c8[j >> 2] |= c << (8 * (j & 3));
          else c8[0] |= c << (4 * j);
        });
      } else if (bits == 8) {
        c8[0] = v == 0 ? packed[0] : v == 1 ? packed[2] : v == 2 ? packed[4] : packed[6];
        c8[1] = v == 0 ? packed[1] : v == 1 ? packed[3] : v == 2 ? packed[5] : packed[7];
      } else {
        c8[0] = v == 0 ? packed[0] : v == 1 ? packed[1] : v == 2 ? packed[2] : packed[3];
        c8[1] = 0u;
      }
      if (bits == 8) reinterpret_cast<uint2*>(cdst)[v] = make_uint2(c8[0], c8[1]);
      else reinterpret_cast<uint32_t*>(cdst)[v] = c8[0];
    }
  }
  if (bad) report(status, KVQ_ERR_NONFINITE);
  *szw = __half_as_ushort(gp.scale_h) |
         (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(static_cast<int>(gp.zf)))) << 16);
}

// Squared quantisation error of one group, sum_i (x_i - x_hat_i)^2 with
// x_hat = (code - z) * s the value the cache would hold at `bits` bits, and
// its squared norm sum_i x_i^2, two values per instruction.  With u and d as
// in quantize_group, x - x_hat = d wherever |d| <= s / 2 and no code is
// clamped (at a tie, |d| = s / 2, either neighbour gives the same error).  A
// quarter with some |d| > s / 2, or a NaN, or a clamped group, is redone with
// code_exact.  Each square-and-add rounds once.
__device__ __forceinline__ float2 group_sq_error(const uint32_t (&w)[16], const uint16_t* src, int bits, bool& bad) {
  const GroupParams gp = group_params(w, bits);
  bad |= gp.bad;
  if (gp.flat) {   // every value 0 (x_hat = 0): no error; a NaN among zeros is reported
    bad |= group_has_nan(w);
    return make_float2(0.0f, 0.0f);
  }
  const float2 r2 = make_float2(gp.rcp, gp.rcp), c2 = make_float2(gp.C, gp.C);
  const float2 nc2 = make_float2(-gp.C, -gp.C), ns2 = make_float2(-gp.sf, -gp.sf);
  const float hs = 0.5f * gp.sf;
  float2 nrm2 = make_float2(0.0f, 0.0f);
  float errq[4];
  unsigned redo = 0;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float2 err2 = make_float2(0.0f, 0.0f);
    float dmax = 0.0f;
#pragma unroll
    for (int k = 4 * v; k < 4 * v + 4; ++k) {
      const float2 x2 = bf16x2_to_float2(w[k]);
      nrm2 = __ffma2_rn(x2, x2, nrm2);
      const float2 d2 = __ffma2_rn(__fadd2_rn(__ffma2_rn(x2, r2, c2), nc2), ns2, x2);
      dmax = fmaxf(dmax, fmaxf(fabsf(d2.x), fabsf(d2.y)));
      err2 = __ffma2_rn(d2, d2, err2);
    }
    errq[v] = __fadd_rn(err2.x, err2.y);
    redo |= (dmax <= hs && errq[v] == errq[v] ? 0u : 1u) << v;   // a NaN makes the sum NaN
  }
  if (group_clamps(gp)) redo = 0xFu;
  if (redo != 0u) {
    const int zero = static_cast<int>(gp.zf);
#pragma unroll 1
    for (int v = 0; v < 4; ++v) {
      if (!((redo >> v) & 1u)) continue;
      float e = 0.0f;
      quarter_values(src, v, [&](int, float x) {
        bad |= x != x;
        const float d = __fmaf_rn(-static_cast<float>(code_exact(x, gp) - zero), gp.sf, x);
        e = __fmaf_rn(d, d, e);
      });
      errq[v] = e;
    }
  }
  return make_float2(__fadd_rn(__fadd_rn(errq[0], errq[1]), __fadd_rn(errq[2], errq[3])),
                     __fadd_rn(nrm2.x, nrm2.y));
}

// resident blocks of 256 threads per SM the register budget is sized for (tunable at build time)
#ifndef KVQ_QUANT_MIN_BLOCKS
#define KVQ_QUANT_MIN_BLOCKS 5
#endif

// One thread per (row, group): row = (b * Hkv + h) * nt + t.  (A persistent
// loop that issued the next group's loads before this group's arithmetic
// measured slower: the extra registers cost more occupancy than it gained.)
// PAGED: the cache is a page pool addressed through p.bt; LENS: rows at
// positions t0 + t >= p.lens[b] are not quantised, and those before the end
// of that length's 128-token tile are cleared (codes and scale/zero word 0,
// which dequantise to exact zeros for the prefill's last tile); separate
// instantiations, so the plain kernel carries none of it.
template <int D, bool PAGED, bool LENS>
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
    if constexpr (LENS) {
      const int len = min(max(p.lens[b], 0), p.Tcap);
      if (p.t0 + t >= len) {
        const int64_t off = p.plane_off[h] + pos * (D * bits / 8) + g * (32 * bits / 8);
        const int64_t si = (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G + g;
        if (p.t0 + t < ((len + 127) & ~127) &&
            group_dst_ok(off, 4 * bits, si, p.codes_bytes, static_cast<int64_t>(p.Hkv) * p.B * p.Tcap * G, p.status)) {
          uint4* dst = reinterpret_cast<uint4*>(p.codes + off);
          dst[0] = make_uint4(0u, 0u, 0u, 0u);
          if (bits == 8) dst[1] = make_uint4(0u, 0u, 0u, 0u);
          p.sz[si] = 0u;
        }
        continue;
      }
    }
    if constexpr (PAGED) {
      const int tl = p.t0 + t;
      if (!KVQ_IN_RANGE(tl / 64 < p.bt_stride, p.status)) continue;
      const int page = p.bt[static_cast<int64_t>(b) * p.bt_stride + tl / 64];
      if (page < 0 || page >= p.B) {   // a page outside the pool: report, write nothing
        if (g == 0) report(p.status, KVQ_ERR_INVALID_ARG);
        continue;
      }
      pos = static_cast<int64_t>(page) * 64 + tl % 64;
    }
    const int64_t off = p.plane_off[h] + pos * (D * bits / 8) + g * (32 * bits / 8);
    const int64_t si = (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G + g;
    if (!group_dst_ok(off, 4 * bits, si, p.codes_bytes, static_cast<int64_t>(p.Hkv) * p.B * p.Tcap * G, p.status))
      continue;
    uint32_t w[16];
    const uint16_t* src = p.x + b * p.sx_b + h * p.sx_h + t * p.sx_t + g * 32;
    load_group(w, src);
    quantize_group(w, src, bits, p.codes + off, p.sz + si, p.status);
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
  int64_t codes_bytes;      // size of each code buffer (the debug build's index checks)
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
      if (!KVQ_IN_RANGE((len - 1) / 64 < p.bt_stride, p.status)) continue;
      const int page = p.bt[static_cast<int64_t>(b) * p.bt_stride + (len - 1) / 64];
      if (page < 0 || page >= p.B) {
        if (job == 0 && h == 0 && g == 0) report(p.status, KVQ_ERR_INVALID_ARG);
        continue;
      }
      pos = static_cast<int64_t>(page) * 64 + (len - 1) % 64;
    }
    const int64_t off = p.plane_off[h] + pos * (D * bits / 8) + g * (32 * bits / 8);
    const int64_t si = (static_cast<int64_t>(h) * p.B * p.Tcap + pos) * G + g;
    if (!group_dst_ok(off, 4 * bits, si, p.codes_bytes, static_cast<int64_t>(p.Hkv) * p.B * p.Tcap * G, p.status))
      continue;
    uint32_t w[16];
    const uint16_t* src = p.x[job] + bh * D + g * 32;
    load_group(w, src);
    quantize_group(w, src, bits, p.codes[job] + off, p.sz[job] + si, p.status);
  }
}

// Per-head error statistics: grid (chunks, H); block (c, h) takes groups
// c * 256 + tid, then every chunks * 256, of head h's B * T * G groups
// (row r = b * T + t, group g), and writes its (error, norm) sums in fp64 to
// part[h][c]; head_stats_reduce adds the chunks in a fixed order, so the
// result does not depend on scheduling.
struct SParams {
  FastDiv div_t;            // r -> (b, t)
  const uint16_t* x;        // bf16 [B][H][T][D]
  const float* w;           // [B][H][T] or null (1)
  const int32_t* lens;      // [B] or null (T)
  double* part;             // [H][chunks][2]
  int32_t* status;
  int32_t B, H, T, bits, chunks;
};

constexpr int kStatThreads = 256;
// Resident blocks the register budget is sized for.  Measured alternatives
// (3, 5 or 6 blocks; two groups per iteration; a register prefetch of the
// next group) were no faster.
constexpr int kStatBlocksPerSM = 4;

template <int D>
__global__ void __launch_bounds__(kStatThreads, kStatBlocksPerSM) head_stats_kernel(const __grid_constant__ SParams p) {
  constexpr int G = D / 32;
  const int h = blockIdx.y;
  // the reduction launched after this kernel may be scheduled now; it waits
  // for this grid's completion before reading the partial sums
  grid_launch_dependents();
  const int64_t n = static_cast<int64_t>(p.B) * p.T * G;
  // (error, norm) summed in fp32 with Kahan's compensation (sum - comp is the
  // running total), widened to fp64 once for the block's reduction
  float2 sum = make_float2(0.0f, 0.0f), comp = make_float2(0.0f, 0.0f);
  const float2 m1 = make_float2(-1.0f, -1.0f);
  bool bad = false;
  auto accumulate = [&](float2 e, float wt) {
    e = __fmul2_rn(e, make_float2(wt, wt));
    const float2 y = __ffma2_rn(comp, m1, e);              // e - comp
    const float2 nsum = __fadd2_rn(sum, y);
    comp = __ffma2_rn(y, m1, __ffma2_rn(sum, m1, nsum));   // (nsum - sum) - y
    sum = nsum;
  };
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStatThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(p.chunks) * kStatThreads) {
    const uint32_t r = static_cast<uint32_t>(i / G);
    const int g = static_cast<int>(i % G);
    const uint32_t b = p.div_t.div(r);
    const int t = static_cast<int>(r - b * p.div_t.d);
    if (p.lens != nullptr && t >= p.lens[b]) continue;
    const int64_t row = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
    uint32_t v[16];
    const uint16_t* src = p.x + row * D + g * 32;
    load_group(v, src);
    accumulate(group_sq_error(v, src, p.bits, bad), p.w != nullptr ? p.w[row] : 1.0f);
  }
  if (bad) report(p.status, KVQ_ERR_NONFINITE);
  // the block's sum in fp32 (a tree of depth 8 over compensated per-thread
  // totals: a few units of 2^-24 relative), then fp64 across blocks (the fp64
  // pipe is narrow, so it is kept out of the per-thread tail)
  float2 tot = __ffma2_rn(comp, m1, sum);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot.x = __fadd_rn(tot.x, __shfl_down_sync(0xffffffffu, tot.x, o));
    tot.y = __fadd_rn(tot.y, __shfl_down_sync(0xffffffffu, tot.y, o));
  }
  __shared__ float2 red[kStatThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = tot;
  __syncthreads();
  if (threadIdx.x == 0) {
    double e = 0.0, m = 0.0;
    for (int k = 0; k < kStatThreads / 32; ++k) { e += static_cast<double>(red[k].x); m += static_cast<double>(red[k].y); }
    double* out = p.part + (static_cast<int64_t>(h) * p.chunks + blockIdx.x) * 2;
    out[0] = e;
    out[1] = m;
  }
}

// One warp per head: stats[h] = the sum of part[h][0 .. chunks) in a fixed order.
__global__ void __launch_bounds__(32) head_stats_reduce(const double* part, int chunks, double* stats) {
  const int h = blockIdx.x, lane = threadIdx.x;
  grid_dependency_wait();   // launched as a dependent of head_stats_kernel
  double e = 0.0, m = 0.0;
  for (int c = lane; c < chunks; c += 32) {
    e += part[(static_cast<int64_t>(h) * chunks + c) * 2];
    m += part[(static_cast<int64_t>(h) * chunks + c) * 2 + 1];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    e += __shfl_xor_sync(0xffffffffu, e, o);
    m += __shfl_xor_sync(0xffffffffu, m, o);
  }
  if (lane == 0) {
    stats[2 * h] = e;
    stats[2 * h + 1] = m;
  }
}

}  // namespace

int head_stats_chunks(int B, int H, int T, int D) {
  const int64_t groups = static_cast<int64_t>(B) * T * (D / 32);
  // one resident wave over all heads
  int64_t c = (static_cast<int64_t>(device_sm_count()) * kStatBlocksPerSM + H - 1) / H;
  const int64_t need = (groups + kStatThreads - 1) / kStatThreads;
  if (c > need) c = need;
  if (c > kHeadStatsMaxChunks) c = kHeadStatsMaxChunks;
  return c < 1 ? 1 : static_cast<int>(c);
}

cudaError_t launch_head_stats(const HeadStatsArgs& a, cudaStream_t stream) {
  SParams p;
  p.div_t = FastDiv::make(static_cast<uint32_t>(a.T));
  p.x = a.x; p.w = a.w; p.lens = a.lens;
  p.part = a.part; p.status = a.status;
  p.B = a.B; p.H = a.H; p.T = a.T; p.bits = a.bits;
  p.chunks = head_stats_chunks(a.B, a.H, a.T, a.D);
  const dim3 grid(static_cast<unsigned>(p.chunks), static_cast<unsigned>(a.H));
  if (a.D == 128) head_stats_kernel<128><<<grid, kStatThreads, 0, stream>>>(p);
  else head_stats_kernel<64><<<grid, kStatThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the fixed-order sum, launched while the statistics kernel still runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.H));
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_stats_reduce, static_cast<const double*>(a.part), p.chunks, a.stats);
}

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream) {
  QParams p;
  p.x = a.x;
  p.sx_b = a.sx_b; p.sx_h = a.sx_h; p.sx_t = a.sx_t;
  p.codes = a.codes; p.sz = a.sz; p.status = a.status;
  p.B = a.B; p.Hkv = a.Hkv; p.Tcap = a.Tcap; p.t0 = a.t0; p.nt = a.nt;
  p.bt = a.bt;
  p.bt_stride = a.bt_max_pages;
  p.lens = a.lens;
  if (p.lens != nullptr && p.bt != nullptr) return cudaErrorInvalidValue;
  p.rows = static_cast<int64_t>(a.bt != nullptr ? a.bt_B : a.B) * a.Hkv * a.nt;
  if (p.rows >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // rows are indexed in 32 bits
  p.codes_bytes = a.layout.off4 + static_cast<int64_t>(a.layout.n4) * a.B * a.Tcap * (a.D / 2);
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
    if (p.bt != nullptr) quantize_kernel<128, true, false><<<g, 256, 0, stream>>>(p);
    else if (p.lens != nullptr) quantize_kernel<128, false, true><<<g, 256, 0, stream>>>(p);
    else quantize_kernel<128, false, false><<<g, 256, 0, stream>>>(p);
  } else {
    if (p.bt != nullptr) quantize_kernel<64, true, false><<<g, 256, 0, stream>>>(p);
    else if (p.lens != nullptr) quantize_kernel<64, false, true><<<g, 256, 0, stream>>>(p);
    else quantize_kernel<64, false, false><<<g, 256, 0, stream>>>(p);
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
  p.codes_bytes = a.layout.off4 + static_cast<int64_t>(a.layout.n4) * a.B * a.Tcap * (a.D / 2);
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
