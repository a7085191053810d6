// kvq_prefill.cu -- prefill attention (causal or not) over the group-quantised KV cache
// on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Method (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》): the score matrix is
// cut into 128x128 tiles and never materialised; each tile's softmax statistics
// (running max, normaliser) are carried forward and a final correction divides
// by the normaliser (§2.2); whole key tiles may be skipped by a block-sparse
// mask (§1.3, §2.3); K and V are read as group-quantised codes -- 8 or 4 bits,
// chosen per KV head (§2.4) -- and dequantised on the fly (§1.3, §2.4).  The
// attention itself is softmax(Q K^T / sqrt(d)) V
// (《一只"兔子"如何搅动大模型推理赛道的底层逻辑》 §3.1), with the causal rule or, for
// non-causal prefill, over every key of the sequence (then the mask may skip
// any off-diagonal tile; query tiles all carry nT key tiles).
//
// One CTA (512 threads, one per SM) computes one 128-row query tile for two
// query heads that share a KV head, so every dequantised K/V tile feeds two
// heads' products:
//   warp 0      allocates TMEM, loads the bf16 Q tiles by TMA, and frees TMEM
//               once every other role is done;
//   warps 1, 2  one elected lane each issues head h = warp - 1's tcgen05.mma:
//                 S_h = Q_h K^T (A, B from shared memory) and
//                 O_h += P_h V   (P from TMEM, V from shared memory), its
//                 first two products (keys 0-31) as soon as the softmax has
//                 stored that chunk of P, the rest once all of P is stored;
//               the heads' products touch disjoint TMEM columns, so each
//               head's chain (S_h, softmax, P_h V, next S_h) runs on its own
//               and the two take turns: head 0's block (P_0 V, next S_0),
//               then head 1's, so that one head's softmax runs while the
//               other's products occupy the tensor pipe; an issuing thread
//               stalls at the pipe's rate, and the turn hand-over replaces the
//               gap a single issuer leaves while it checks the next head's
//               barriers;
//   warps 4-7   convert Q to fp16 in place, then per kept key tile load the
//               codes and fp16 scale/zero words into registers one tile part
//               (K or V) ahead of their use and write exact-rounded fp16
//               K_hat = (c - z) * s and V_hat tiles in the 128-byte-swizzled
//               layout the tensor core reads (2 stages); which row and chunk
//               each lane takes is chosen per code format so that a warp's
//               loads cover whole contiguous rows and every 8-lane phase of a
//               16-byte store covers all 32 banks;
//   warps 8-11  softmax of head 0, warps 12-15 softmax of head 1: one thread
//               per query row reads its S row from TMEM (two passes of four
//               32-column loads, the next load in flight while a chunk is
//               worked on), applies the causal rule on the diagonal tile
//               (causal only), updates (max, sum) in the log2 domain with
//               two-wide fp32 arithmetic, writes P (fp16) back over S, and at
//               the end scales O by 1 / sum and stores it.
// TMEM (512 columns): S_0 [0,128) O_0 [128,128+D) S_1 [256,384) O_1 [384,384+D).
// The running max is only moved (and O rescaled) when it grows by more than
// 2^8, so P stays <= 256 and rescales are rare; the final division uses the
// sum accumulated against the same max, which keeps the result exact.
//
// 4-bit heads: a code byte holds channels 2i (low nibble) and 2i+1.  Within
// each 8-channel block the fp16 tiles hold the channels in the order
// 0,4,1,5,2,6,3,7 (what one shift and one mask per pair of values give); Q
// gets the same order when it is converted, so Q.K is unchanged, and O's
// columns come out in that order and are put back in the epilogue.
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kT = 128;           // tile edge (query rows, keys)
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSub = 2048;        // code bytes one dequant iteration reads: 128 threads x 16 B

struct PParams {
  CUtensorMap tm_q;               // bf16 [B*Hq*S][D], box [64][128], 128B swizzle
  const uint8_t* kcodes;          // code buffer of the K cache (every head's plane)
  const uint8_t* vcodes;
  const uint32_t* ksz;
  const uint32_t* vsz;
  const uint8_t* tile_mask;       // [nT][nT] or null
  void* out;
  int32_t* status;
  int32_t out_dtype;
  int32_t B, Hq, Hkv, S, Tcap, rep, pairs, nT;
  int32_t causal;                 // 1: keys j <= i; 0: every key of the sequence
  const int32_t* lens;            // [B] sequence lengths (<= S) or null (every sequence S long)
  float scale_log2;
  uint64_t wait_ns;               // bounded-wait limit
  int32_t issue_limit;            // test only: 0 withholds the query load (every first wait then runs out)
  int64_t plane_off[KVQ_MAX_HKV]; // byte offset of each KV head's code plane
  int64_t codes_bytes;            // size of each code buffer (the debug build's index checks)
  int8_t bits[KVQ_MAX_HKV];       // 8 or 4 per KV head
};

// barriers
enum {
  B_QFULL = 0, B_QREADY, B_KFULL0, B_KFULL1, B_VFULL0, B_VFULL1, B_KVEMPTY0, B_KVEMPTY1,
  B_SFULL0, B_SFULL1, B_PFIRST0, B_PFIRST1, B_PFULL0, B_PFULL1, B_ORDY0, B_ORDY1, B_MMADONE, B_TURN0, B_TURN1,
  B_EXIT, B_COUNT
};
// Every warp but warp 0 arrives once on B_EXIT when it is done with shared
// memory, TMEM and its asynchronous operations, on the normal path and after
// a timed-out wait alike; warp 0 frees TMEM only after that.
constexpr int kExitArrivals = kThreads / 32 - 1;

// shared memory layout (bytes from a 1024-aligned base)
template <int D>
struct PLayout {
  static constexpr int kQBytes = kT * D * 2;            // one head's fp16 tile: D/64 blocks of [128 rows][128 B]
  static constexpr int kOffQ = 0;                       // 2 heads
  static constexpr int kOffK = kOffQ + 2 * kQBytes;     // 2 stages
  static constexpr int kOffV = kOffK + 2 * kQBytes;     // 2 stages
  static constexpr int kOffBar = kOffV + 2 * kQBytes;
  static constexpr int kOffTmem = kOffBar + B_COUNT * 8;
  static constexpr int kBytes = kOffTmem + 16 + 1024;
};
static_assert(PLayout<128>::kBytes <= 232448, "shared memory of the D = 128 prefill");

// How the dequant warpgroup walks one code tile (the K or V part of a key
// tile) of a (D, BITS) head.  Iteration `it` covers RPI token rows of R
// bytes (2 KB), 16 bytes per thread; a 16-byte chunk holds VPC channels (16
// or 32) and becomes two or four 16-byte fp16 chunks of the swizzled operand
// tile.
template <int D, int BITS>
struct DqFmt {
  static constexpr int R = D * BITS / 8;     // code bytes per token row
  static constexpr int RPI = kSub / R;       // rows per iteration
  static constexpr int NI = kT / RPI;        // iterations (ring sub-chunks) per part
  static constexpr int VPC = 128 / BITS;     // channels per chunk
  static_assert(RPI * NI == kT, "whole iterations per part");
};

// Row (within an iteration) and chunk of the 16 code bytes thread t loads.
// A warp's 32 lanes cover whole consecutive rows (512 contiguous bytes).
// With the 128-byte swizzle, fp16 chunk x of row r sits at bank group
// x ^ (r & 7), and the D/64 blocks of a tile are 16 KB apart (the same
// banks).  Per format, the eight lanes of each store phase take:
//   8-bit, D 128: one half (64 B) of row r and the other half of row r + 1,
//                 so the stores (two chunks per lane) go to even chunk
//                 indices in one row and odd ones in the other;
//   4-bit, D 128: rows r .. r+3 (r a multiple of 4), the first 32 bytes of
//                 rows r, r+3 and the last 32 of rows r+1, r+2 (or the other
//                 way round): each store phase writes the four swizzle rows
//                 of a quad, once in the low and once in the high half of the
//                 chunk index;
//   D 64:         two (8-bit) or four (4-bit) whole consecutive rows.
template <int D, int BITS>
__device__ __forceinline__ void dq_lane(int t, int& row, int& c) {
  const int w = t >> 5, l = t & 31;
  if constexpr (D == 128 && BITS == 8) {
    const int sub = (l & 7) >> 2, ph = (l >> 3) & 1;
    row = 4 * w + 2 * (l >> 4) + sub;
    c = (l & 3) + 4 * (sub ^ ph);
  } else if constexpr (D == 128 && BITS == 4) {
    const int rr = (l & 7) >> 1, ph = (l >> 3) & 1;
    const int hi = (rr ^ (rr >> 1)) & 1;     // rows 1, 2 of the quad take the other half
    row = 8 * w + 4 * (l >> 4) + rr;
    c = 2 * (hi ^ ph) + (l & 1);
  } else if constexpr (BITS == 8) {          // D 64
    row = t >> 2;
    c = t & 3;
  } else {
    row = t >> 1;
    c = t & 1;
  }
}

__device__ __forceinline__ bool tile_kept(const PParams& p, int qt, int kt) {
  return kt == qt || p.tile_mask == nullptr || p.tile_mask[qt * p.nT + kt] != 0;
}

// key tiles [0, kt_end) of query tile qt can take part (L: the sequence's length)
__device__ __forceinline__ int key_tile_end(const PParams& p, int qt, int L) {
  return p.causal ? qt + 1 : (L + kT - 1) / kT;
}

__device__ __forceinline__ int next_kept(const PParams& p, int qt, int kt, int end) {
  while (kt < end && !tile_kept(p, qt, kt)) ++kt;
  return kt;
}

// two-wide fp32 arithmetic (one instruction for a pair of values)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "add.f32x2 rd, rd, ra;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 16 bytes to a shared-window address
__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// One code chunk (16 bytes, channels ch0 ..) -> OC fp16 chunks of (c - z) * s
// (exact difference, one rounding) in the 128-byte-swizzled K-major tile
// [D/64 blocks][128 rows][128 B] at dst.
template <int BITS>
__device__ __forceinline__ void dequant_chunk(uint32_t dst, int row, int ch0, uint4 w, uint32_t word) {
  constexpr int OC = BITS == 8 ? 2 : 4;
  const uint32_t zb = zero_biased2(word);
  const uint32_t s2 = (word & 0xFFFFu) | (word << 16);
  // 4-bit high nibbles: c - z = (1024 + 16 c) / 16 - 64 - z in one exact FMA
  const uint32_t mz = hsub2_u32(0x63806380u /* (960, 960) */, zb);   // -(64 + z), exact
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[4 * OC];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BITS == 8) {
      // channels 4i .. 4i + 3 in order
      o[2 * i] = hmul2_u32(hsub2_u32(bytes01_biased(wv[i]), zb), s2);
      o[2 * i + 1] = hmul2_u32(hsub2_u32(bytes23_biased(wv[i]), zb), s2);
    } else {
      // channels 8i .. 8i + 7 in the order 0,4,1,5,2,6,3,7
      const uint32_t w8 = wv[i] >> 8;
      o[4 * i + 0] = hmul2_u32(hsub2_u32(nib_biased(wv[i]), zb), s2);
      o[4 * i + 1] = hmul2_u32(hfma2_u32((wv[i] & 0x00F000F0u) | 0x64006400u, kHalf2Sixteenth, mz), s2);
      o[4 * i + 2] = hmul2_u32(hsub2_u32(nib_biased(w8), zb), s2);
      o[4 * i + 3] = hmul2_u32(hfma2_u32((w8 & 0x00F000F0u) | 0x64006400u, kHalf2Sixteenth, mz), s2);
    }
  }
  const int kb = ch0 >> 6, cb = (ch0 & 63) >> 3, sw = row & 7;
  const uint32_t rowp = dst + kb * (kT * 128) + row * 128;
#pragma unroll
  for (int i = 0; i < OC; ++i) sts128(rowp + (((cb + i) ^ sw) << 4), o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// One part (K or V) of a key tile in a dequant thread's registers: its code
// chunk and scale/zero word of every iteration.
template <int D, int BITS>
struct PartRegs {
  uint4 c[DqFmt<D, BITS>::NI];
  uint32_t w[DqFmt<D, BITS>::NI];
};

// (cend, send, status: the ends of the code and scale/zero buffers for the
// debug build's index checks; a failed check loads zeros instead)
template <int D, int BITS>
__device__ __forceinline__ void load_part(PartRegs<D, BITS>& r, const uint8_t* codes, const uint32_t* sz, int kt,
                                          int row, int c, int g, const uint8_t* cend, const uint32_t* send,
                                          int32_t* status) {
  using F = DqFmt<D, BITS>;
  constexpr int G = D / 32;
#pragma unroll
  for (int it = 0; it < F::NI; ++it) {
    const size_t tok = static_cast<size_t>(kt) * kT + F::RPI * it + row;
    const uint8_t* cp = codes + tok * F::R + c * 16;
    const uint32_t* sp = sz + tok * G + g;
    if (KVQ_IN_RANGE(cp + 16 <= cend && sp < send, status)) {
      r.c[it] = __ldg(reinterpret_cast<const uint4*>(cp));
      r.w[it] = __ldg(sp);
    } else {
      r.c[it] = make_uint4(0u, 0u, 0u, 0u);
      r.w[it] = 0u;
    }
  }
}

template <int D, int BITS>
__device__ __forceinline__ void store_part(uint32_t dst, const PartRegs<D, BITS>& r, int row, int c) {
  using F = DqFmt<D, BITS>;
#pragma unroll
  for (int it = 0; it < F::NI; ++it) dequant_chunk<BITS>(dst, F::RPI * it + row, c * F::VPC, r.c[it], r.w[it]);
}

// Dequant warpgroup after Q: every kept key tile's K and V parts into the
// two-stage fp16 operand tiles.  Two register sets: while one part is
// converted, the next part's codes are on their way from L2 / HBM.  Returns
// early (warp-uniformly) if a wait runs out.
template <int D, int BITS>
__device__ __forceinline__ void dequant_loop(const PParams& p, uint8_t* smem, uint64_t* bar, int b, int kvh, int qt,
                                             int kt_end, int t, int lane) {
  using L = PLayout<D>;
  using F = DqFmt<D, BITS>;
  int row, c;
  dq_lane<D, BITS>(t, row, c);
  const int g = c * F::VPC / 32;
  const size_t base_tok = static_cast<size_t>(b) * p.Tcap;
  const uint8_t* kcodes = p.kcodes + p.plane_off[kvh] + base_tok * F::R;
  const uint8_t* vcodes = p.vcodes + p.plane_off[kvh] + base_tok * F::R;
  const size_t szrow = (static_cast<size_t>(kvh) * p.B + b) * p.Tcap;
  const uint32_t* ksz = p.ksz + szrow * (D / 32);
  const uint32_t* vsz = p.vsz + szrow * (D / 32);
  const int64_t sz_words = static_cast<int64_t>(p.Hkv) * p.B * p.Tcap * (D / 32);
  const uint8_t* kcend = p.kcodes + p.codes_bytes;
  const uint8_t* vcend = p.vcodes + p.codes_bytes;
  const uint32_t* ksend = p.ksz + sz_words;
  const uint32_t* vsend = p.vsz + sz_words;
  const uint32_t kdst = smem_u32(smem + L::kOffK);
  const uint32_t vdst = smem_u32(smem + L::kOffV);
  PartRegs<D, BITS> ra, rb;
  int kt = next_kept(p, qt, 0, kt_end);
  if (kt < kt_end) load_part<D, BITS>(ra, kcodes, ksz, kt, row, c, g, kcend, ksend, p.status);
  for (int j = 0; kt < kt_end; ++j) {
    const int st = j & 1;
    const int kt_next = next_kept(p, qt, kt + 1, kt_end);
    load_part<D, BITS>(rb, vcodes, vsz, kt, row, c, g, vcend, vsend, p.status);
    if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&bar[B_KVEMPTY0 + st], ((j >> 1) - 1) & 1, p.status, p.wait_ns)))
      return;
    store_part<D, BITS>(kdst + st * L::kQBytes, ra, row, c);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_KFULL0 + st]);
    if (kt_next < kt_end) load_part<D, BITS>(ra, kcodes, ksz, kt_next, row, c, g, kcend, ksend, p.status);
    store_part<D, BITS>(vdst + st * L::kQBytes, rb, row, c);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_VFULL0 + st]);
    kt = kt_next;
  }
}

// Zeros in the output rows of this work item (a query tile past its sequence's end).
template <int D>
__device__ __forceinline__ void zero_out_tile(const PParams& p, int b, int h0, int nh, int qt) {
  const size_t row0 = (static_cast<size_t>(b) * p.Hq + h0) * p.S + static_cast<size_t>(qt) * kT;
  const int esz = p.out_dtype == KVQ_OUT_F32 ? 4 : 2;
  const int vec_per_row = D * esz / 16;
  if (!KVQ_IN_RANGE(row0 + static_cast<size_t>(nh - 1) * p.S + kT <= static_cast<size_t>(p.B) * p.Hq * p.S, p.status))
    return;
  for (int h = 0; h < nh; ++h) {
    uint4* base =
        reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (row0 + static_cast<size_t>(h) * p.S) * D * esz);
    for (int i = threadIdx.x; i < kT * vec_per_row; i += kThreads) base[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// 32 output values of one row (TMEM columns 32c .. 32c+31, times inv) to global memory.
template <int D>
__device__ __forceinline__ void store_row32(const PParams& p, size_t off, const float (&o)[32]) {
  if (!KVQ_IN_RANGE(off + 32 <= static_cast<size_t>(p.B) * p.Hq * p.S * D, p.status)) return;
  if (p.out_dtype == KVQ_OUT_F32) {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 t2 = __floats2bfloat162_rn(o[8 * i + 2 * e], o[8 * i + 2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&t2);
      }
      dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PParams p) {
  using L = PLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: (query tile, b, kv head, head pair), longest (last) query tiles first ----
  const int per_qt = p.B * p.Hkv * p.pairs;
  const int qt = p.nT - 1 - static_cast<int>(blockIdx.x) / per_qt;
  int rem = static_cast<int>(blockIdx.x) % per_qt;
  const int pair = rem % p.pairs; rem /= p.pairs;
  const int kvh = rem % p.Hkv;
  const int b = rem / p.Hkv;
  const int h0 = kvh * p.rep + 2 * pair;
  const int nh = (2 * pair + 1 < p.rep) ? 2 : 1;
  const bool four = p.bits[kvh] == 4;
  // the sequence's length: a query tile wholly past it writes zeros and ends
  // here, before any barrier or TMEM is set up (the decision is the CTA's own)
  int Ls = p.S;
  if (p.lens != nullptr) {
    Ls = p.lens[b];
    if (Ls < 0 || Ls > p.S) {
      if (threadIdx.x == 0 && qt == 0) report(p.status, KVQ_ERR_INVALID_ARG);
      Ls = min(max(Ls, 0), p.S);
    }
  }
  if (qt * kT >= Ls) {
    zero_out_tile<D>(p, b, h0, nh, qt);
    return;
  }
  const int q_valid = min(kT, Ls - qt * kT);   // query rows of this tile inside the sequence

  if (threadIdx.x == 0) {
    mbar_init(&bar[B_QFULL], 1);
    mbar_init(&bar[B_QREADY], 4);
    mbar_init(&bar[B_KFULL0], 4); mbar_init(&bar[B_KFULL1], 4);
    mbar_init(&bar[B_VFULL0], 4); mbar_init(&bar[B_VFULL1], 4);
    mbar_init(&bar[B_KVEMPTY0], nh); mbar_init(&bar[B_KVEMPTY1], nh);
    mbar_init(&bar[B_SFULL0], 1); mbar_init(&bar[B_SFULL1], 1);
    mbar_init(&bar[B_PFIRST0], 4); mbar_init(&bar[B_PFIRST1], 4);
    mbar_init(&bar[B_PFULL0], 4); mbar_init(&bar[B_PFULL1], 4);
    mbar_init(&bar[B_ORDY0], 1); mbar_init(&bar[B_ORDY1], 1);
    mbar_init(&bar[B_MMADONE], nh);
    mbar_init(&bar[B_TURN0], 1); mbar_init(&bar[B_TURN1], 1);
    mbar_init(&bar[B_EXIT], kExitArrivals);
    fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Registers: the CTA is launched with 128 per thread (checked on the host).
  // Each warpgroup resets its own limit at the top of its branch:
  //   TMA/MMA 128 -> 80 (frees 6144), softmax x2 128 -> 120 (frees 2048),
  //   dequant 128 -> 192 (takes 8192): 128 x (80 + 192 + 120 + 120) = 65536
  // = 512 x 128, and per sub-partition (one warp of each warpgroup)
  // 32 x (80 + 192 + 120 + 120) = 16384, its whole register file.

  // number of kept key tiles (identical in every role)
  const int kt_end = key_tile_end(p, qt, Ls);
  int n_kept = kt_end;
  if (p.tile_mask != nullptr) {
    // 16 mask bytes per load where the row allows it; the diagonal counts as
    // kept whatever its byte says
    const uint8_t* row = p.tile_mask + static_cast<size_t>(qt) * p.nT;
    n_kept = 0;
    int kt = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
      for (; kt + 16 <= kt_end; kt += 16) {
        const uint4 m4 = *reinterpret_cast<const uint4*>(row + kt);
        const uint32_t w4[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)   // bytes that are not zero: their top bit after adding 0x7F to the low seven
          n_kept += __popc((((w4[i] & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w4[i]) & 0x80808080u);
      }
    }
    for (; kt < kt_end; ++kt) n_kept += row[kt] != 0 ? 1 : 0;
    if (qt < kt_end && row[qt] == 0) ++n_kept;
  }
  const uint64_t wns = p.wait_ns;

  if (warp < 4) {
  tc::reg_dealloc<80>();
  if (warp == 0) {
    // ---------------- Q by TMA, then free TMEM once every role is done ----------------
    const bool issue = p.issue_limit != 0;
    if (lane == 0 && issue) {
      mbar_arrive_expect_tx(&bar[B_QFULL], nh * L::kQBytes);
      for (int h = 0; h < nh; ++h) {
        const int32_t y = ((b * p.Hq + h0 + h) * p.S) + qt * kT;
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb)
          tma_2d_g2s(smem + L::kOffQ + h * L::kQBytes + kb * (kT * 128), &p.tm_q, 64 * kb, y, &bar[B_QFULL]);
      }
    }
    __syncwarp();
    // The other roles finish in bounded time: each stops at its first wait
    // that runs out, and a role waits at most a few times per kept key tile.
    // So the exit wait gets a deadline of that many limits.
    const uint64_t deadline = wns * static_cast<uint64_t>(4 * n_kept + 8);
    const uint64_t t0 = global_ns();
    uint32_t n = 0;
    while (!mbar_try_wait(&bar[B_EXIT], 0)) {
      if ((++n & 255u) == 0 && global_ns() - t0 > deadline) {
        report(p.status, KVQ_ERR_TIMEOUT);
        break;
      }
    }
    // the query copy has landed before the CTA can exit (normally long since)
    if (lane == 0 && issue) mbar_wait(&bar[B_QFULL], 0, p.status, wns);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
    return;
  }

  if (warp == 1 || warp == 2) {
    // ---------------- MMA issuers, one warp per head ----------------
    // Every lane runs the waits (their outcome is made warp-uniform) and the
    // descriptor arithmetic; the elected lane -- lane 0, the lowest of a
    // converged warp -- issues the products, their commits and the turn
    // hand-overs, so every commit tracks every product of this head.
    const int h = warp - 1;
    if (h >= nh) {
      if (lane == 0) mbar_arrive(&bar[B_EXIT]);
      return;
    }
    const uint32_t id_qk = tc::idesc_f16_f32(kT, kT, false);
    const uint32_t id_pv = tc::idesc_f16_f32(kT, D, true);
    const uint32_t qh = smem_u32(smem + L::kOffQ) + h * L::kQBytes;
    const uint32_t k_base = smem_u32(smem + L::kOffK);
    const uint32_t v_base = smem_u32(smem + L::kOffV);
    const uint32_t d_s = tmem + h * 256, d_o = d_s + 128;
    auto wait_all = [&](int which, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(&bar[which], parity, p.status, wns));
    };
    // S_h = Q_h K^T over the K tile in stage st (elected lane)
    auto issue_qk = [&](int st) {
      const uint32_t kh = k_base + st * L::kQBytes;
      tc::mma_ss<false>(d_s, tc::smem_desc_sw128(qh, 16, 1024), tc::smem_desc_sw128(kh, 16, 1024), id_qk);
#pragma unroll
      for (int s = 1; s < D / 16; ++s) {
        const uint32_t off = (s >> 2) * (kT * 128) + (s & 3) * 32;
        tc::mma_ss<true>(d_s, tc::smem_desc_sw128(qh + off, 16, 1024), tc::smem_desc_sw128(kh + off, 16, 1024), id_qk);
      }
      tc::commit(&bar[B_SFULL0 + h]);
    };
    // O_h (+)= P_h V over part `hf` of the V tile in stage st (elected lane):
    // keys 0-31, as soon as the softmax has stored that much of P, then keys
    // 32-127
    auto issue_pv = [&](int st, bool first, int hf) {
      const uint32_t vs = v_base + st * L::kQBytes;
      if (hf == 0) {
        const uint64_t v0 = tc::smem_desc_sw128(vs, kT * 128, 1024);
        if (first) tc::mma_ts<false>(d_o, d_s, v0, id_pv);
        else tc::mma_ts<true>(d_o, d_s, v0, id_pv);
      }
#pragma unroll
      for (int s = hf == 0 ? 1 : 2; s < (hf == 0 ? 2 : kT / 16); ++s)
        tc::mma_ts<true>(d_o, d_s + s * 8, tc::smem_desc_sw128(vs + s * 2048, kT * 128, 1024), id_pv);
    };
    // Turns: block b = -1 is Q.K^T of tile 0, block b >= 0 is P.V of tile b
    // and Q.K^T of tile b + 1.  With two heads, head 0 issues block b after
    // head 1's block b - 1 (completion b of B_TURN0) and head 1 after head 0's
    // block b (completion b + 1 of B_TURN1).
    const bool turns = nh == 2;
    auto take_turn = [&](int blk) -> bool {
      if (!turns || (h == 0 && blk < 0)) return true;
      return h == 0 ? wait_all(B_TURN0, blk & 1) : wait_all(B_TURN1, (blk + 1) & 1);
    };
    auto pass_turn = [&]() {
      if (turns) mbar_arrive(&bar[h == 0 ? B_TURN1 : B_TURN0]);
    };
    bool ok = wait_all(B_QREADY, 0) && (n_kept == 0 || (wait_all(B_KFULL0, 0) && take_turn(-1)));
    tc::fence_after_sync();
    if (ok && n_kept > 0) {
      if (tc::elect_one()) {
        issue_qk(0);
        pass_turn();
      }
      __syncwarp();
    }
    for (int j = 0; j < n_kept && ok; ++j) {
      const int st = j & 1;
      ok = wait_all(B_VFULL0 + st, (j >> 1) & 1) && wait_all(B_PFIRST0 + h, j & 1) && take_turn(j);
      if (!ok) break;
      tc::fence_after_sync();
      if (tc::elect_one()) issue_pv(st, j == 0, 0);   // while the softmax writes the rest of P
      __syncwarp();
      ok = wait_all(B_PFULL0 + h, j & 1);
      if (!ok) break;
      tc::fence_after_sync();
      if (tc::elect_one()) {
        issue_pv(st, false, 1);
        tc::commit(&bar[B_ORDY0 + h]);
        // this head is done with the stage: its Q.K^T of tile j was issued
        // before this P.V (an issuer's products complete in issue order)
        tc::commit(&bar[B_KVEMPTY0 + st]);
      }
      __syncwarp();
      if (j + 1 < n_kept) {
        // the next K tile is written once both heads' P.V of tile j - 1 are
        // done; this head's P.V queued above covers most of that wait
        ok = wait_all(B_KFULL0 + ((j + 1) & 1), ((j + 1) >> 1) & 1);
        if (!ok) break;
        tc::fence_after_sync();
      }
      if (tc::elect_one()) {
        if (j + 1 < n_kept) issue_qk((j + 1) & 1);
        pass_turn();
      }
      __syncwarp();
    }
    // every product this warp issued has completed (a commit with none
    // pending arrives at once) before the warp reports that it is done
    if (tc::elect_one()) tc::commit(&bar[B_MMADONE]);
    __syncwarp();
    wait_all(B_MMADONE, 0);
    tc::fence_before_sync();
    if (lane == 0) mbar_arrive(&bar[B_EXIT]);
    return;
  }

  if (lane == 0) mbar_arrive(&bar[B_EXIT]);   // warp 3: no role
  return;
  }

  if (warp < 8) {
    tc::reg_alloc<192>();
    // ---------------- dequant warpgroup ----------------
    const int t = threadIdx.x - 128;
    do {
    if (!__all_sync(0xffffffffu, mbar_wait(&bar[B_QFULL], 0, p.status, wns))) break;
    // Q to fp16 in place (exact for bf16 values in fp16 range); for a 4-bit
    // head each 8-channel block in the order 0,4,1,5,2,6,3,7 of the K tiles
    bool finite = true;
    for (int i = t; i < nh * L::kQBytes / 16; i += 128) {
      uint4* ptr = reinterpret_cast<uint4*>(smem + L::kOffQ) + i;
      if (q_valid < kT && ((i & 1023) >> 3) >= q_valid) {   // row past the sequence's end
        *ptr = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      uint4 v = *ptr;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
        finite &= fabsf(lo) < 65504.0f && fabsf(hi) < 65504.0f;
        w[e] = pack_half2(lo, hi);
      }
      if (four) {
        const uint32_t a = prmt(w[0], w[2], 0x5410u), bb = prmt(w[0], w[2], 0x7632u);
        const uint32_t c = prmt(w[1], w[3], 0x5410u), d = prmt(w[1], w[3], 0x7632u);
        w[0] = a; w[1] = bb; w[2] = c; w[3] = d;
      }
      *ptr = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (!finite) report(p.status, KVQ_ERR_NONFINITE);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_QREADY]);
    // Positions past a shorter sequence's end within its last tile read as
    // zeros: the quantiser cleared them (codes and scale/zero words 0), so a
    // masked score (P = 0) never meets a non-finite V_hat in the P.V product.
    if (four) dequant_loop<D, 4>(p, smem, bar, b, kvh, qt, kt_end, t, lane);
    else dequant_loop<D, 8>(p, smem, bar, b, kvh, qt, kt_end, t, lane);
    } while (0);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_EXIT]);
    return;
  }

  // ---------------- softmax warpgroups ----------------
  tc::reg_dealloc<120>();
  const int h = (warp - 8) >> 2;            // head slot 0 or 1
  if (h >= nh) {
    if (lane == 0) mbar_arrive(&bar[B_EXIT]);
    return;
  }
  const int q4 = warp & 3;                  // TMEM lane quarter
  const int r = q4 * 32 + lane;             // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + h * 256;
  const uint32_t o_addr = s_addr + 128;
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY, l_run = 0.0f;
  bool ok = true;
  int j = 0;
  for (int kt = 0; kt < kt_end && ok; ++kt) {
    if (!tile_kept(p, qt, kt)) continue;
    // columns past `lim` are masked: the element-wise causal rule on the
    // diagonal tile, the sequence's end on the last key tile of non-causal
    // prefill (causal rows inside the sequence never reach past it)
    bool masked = p.causal && kt == qt;
    int lim = r;
    if (!p.causal) {
      const int climit = min(kT, Ls - kt * kT);
      masked = climit < kT;
      lim = climit - 1;
    }
    // a timed-out wait ends the loop for the whole warp (its TMEM accesses are warp-wide)
    ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL0 + h], j & 1, p.status, wns));
    if (!ok) break;
    tc::fence_after_sync();
    // pass 1: row max (three-input max, two chains).  Unmasked tiles keep the
    // next 32-column chunk's TMEM load in flight while a chunk is reduced
    // (two register buffers), so only the first load's latency is exposed.
    float mxa = -INFINITY, mxb = -INFINITY;
    if (!masked) {
      uint32_t va[32], vb[32];
      auto mx_chunk = [&](const uint32_t (&v)[32]) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          mxa = fmax3(mxa, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
          mxb = fmax3(mxb, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
      };
      tc::ld_32x32b_x32(s_addr, va);
      tc::wait_ld(va);
      tc::ld_32x32b_x32(s_addr + 32, vb);
      mx_chunk(va);
      tc::wait_ld(vb);
      tc::ld_32x32b_x32(s_addr + 64, va);
      mx_chunk(vb);
      tc::wait_ld(va);
      tc::ld_32x32b_x32(s_addr + 96, vb);
      mx_chunk(va);
      tc::wait_ld(vb);
      mx_chunk(vb);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::ld_32x32b_x32(s_addr + c * 32, v);
        tc::wait_ld(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) mxa = (c * 32 + i > lim) ? mxa : fmaxf(mxa, __uint_as_float(v[i]));
      }
    }
    const float m_tile = fmaxf(mxa, mxb) * sl2;
    float m_use = m_run, alpha = 1.0f;
    if (m_run == -INFINITY || m_tile > m_run + kRescaleThreshold) {
      m_use = fmaxf(m_run, m_tile);
      alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_use);
      m_run = m_use;
    }
    // rescale O (rare) before any P.V of this tile is issued: the previous
    // P.V has finished (it was issued before the Q.K^T that made this S, and
    // an issuer's products complete in order), so the wait returns at once
    if (__any_sync(0xffffffffu, alpha != 1.0f) && j > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_ORDY0 + h], (j - 1) & 1, p.status, wns));
      if (!ok) break;
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tc::ld_32x32b_x32(o_addr + c * 32, v);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tc::st_32x32b_x32(o_addr + c * 32, v);
      }
    }
    // P's first chunk (keys 0-31, and any rescaled O) is stored: the issuer
    // may start this tile's P.V on it while the rest is computed
    auto p_first = [&]() {
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_PFIRST0 + h]);
    };
    // pass 2: P = 2^(S*scale_log2 - m) as fp16 pairs, written over the part of S
    // already read (columns 16c.. of P after S columns 32c.. were loaded);
    // the exponent arguments and the row sum two at a time
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
    const float neg_m = -m_use;
    if (!masked) {
      // P of chunk c goes to columns 16c.. (S columns already read); the next
      // chunk's load is in flight meanwhile, as in pass 1
      uint32_t va[32], vb[32];
      auto p_chunk = [&](const uint32_t (&v)[32], int c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float x0, x1, x2, x3;
          ffma2(x0, x1, __uint_as_float(v[i]), __uint_as_float(v[i + 1]), sl2, neg_m);
          ffma2(x2, x3, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]), sl2, neg_m);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2), p3 = fast_exp2(x3);
          fadd2(s0, s1, p0, p1);
          fadd2(s2, s3, p2, p3);
          pk[i / 2] = pack_half2(p0, p1);
          pk[i / 2 + 1] = pack_half2(p2, p3);
        }
        tc::st_32x32b_x16(s_addr + c * 16, pk);
      };
      tc::ld_32x32b_x32(s_addr, va);
      tc::wait_ld(va);
      tc::ld_32x32b_x32(s_addr + 32, vb);
      p_chunk(va, 0);
      p_first();
      tc::wait_ld(vb);
      tc::ld_32x32b_x32(s_addr + 64, va);
      p_chunk(vb, 1);
      tc::wait_ld(va);
      tc::ld_32x32b_x32(s_addr + 96, vb);
      p_chunk(va, 2);
      tc::wait_ld(vb);
      p_chunk(vb, 3);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        uint32_t pk[16];
        tc::ld_32x32b_x32(s_addr + c * 32, v);
        tc::wait_ld(v);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = (c * 32 + i > lim) ? 0.0f : fast_exp2(fmaf(__uint_as_float(v[i]), sl2, neg_m));
          const float p1 = (c * 32 + i + 1 > lim) ? 0.0f : fast_exp2(fmaf(__uint_as_float(v[i + 1]), sl2, neg_m));
          fadd2(s0, s1, p0, p1);
          pk[i / 2] = pack_half2(p0, p1);
        }
        tc::st_32x32b_x16(s_addr + c * 16, pk);
        if (c == 0) p_first();
      }
    }
    const float psum = (s0 + s1) + (s2 + s3);
    l_run = l_run * alpha + psum;
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_PFULL0 + h]);
    ++j;
  }
  // epilogue: O / l (skipped after a timed-out wait: the output is then unspecified)
  if (ok && n_kept > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_ORDY0 + h], (n_kept - 1) & 1, p.status, wns));
  tc::fence_after_sync();
  // rows past the sequence's end are written as zeros
  const float inv = (l_run > 0.0f && r < q_valid) ? 1.0f / l_run : 0.0f;
  const size_t orow = (static_cast<size_t>(b) * p.Hq + h0 + h) * p.S + static_cast<size_t>(qt) * kT + r;
  if (ok) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tc::ld_32x32b_x32(o_addr + c * 32, v);
      tc::wait_ld();
      float o[32];
      if (four) {
        // column 8m + 2k holds channel 8m + k, column 8m + 2k + 1 channel 8m + 4 + k
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[(i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1)]) * inv;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]) * inv;
      }
      store_row32<D>(p, orow * D + c * 32, o);
    }
  }
  tc::wait_st();   // P and rescaled O stores of a loop left early have landed
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bar[B_EXIT]);
}

// Per device and head dim, set once under a lock: the kernel's large dynamic
// shared memory limit, and whether it was built with the 128 registers per
// thread that the register split above assumes.  1 = ready, -2 = not usable,
// 0 = not yet set.
std::mutex g_prep_mu;
int g_prep[64][2] = {};

template <int D>
int prepare_prefill_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(g_prep_mu);
  int& st = g_prep[dev][D == 128 ? 1 : 0];
  if (st == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, prefill_kernel<D>) != cudaSuccess || fa.numRegs != 128) {
      st = -2;   // unsupported build
    } else if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    PLayout<D>::kBytes) != cudaSuccess) {
      return -1;   // a CUDA error; try again on the next call
    } else {
      st = 1;
    }
  }
  return st;
}

template <int D>
kvq_status launch_prefill_d(const PParams& p, int64_t items, cudaStream_t stream) {
  const int prep = prepare_prefill_on_current_device<D>();
  if (prep == -2) return KVQ_ERR_UNSUPPORTED;
  if (prep != 1) return KVQ_ERR_CUDA;
  prefill_kernel<D><<<static_cast<unsigned>(items), kThreads, PLayout<D>::kBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

kvq_status launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PParams p;
  memset(&p, 0, sizeof(p));
  const int D = a.D;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Hq * a.S;
  if (qrows >= (uint64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (encode_tensor_map_2d(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, D, qrows, D * 2, 64, kT,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return KVQ_ERR_CUDA;
  p.kcodes = a.k->codes;
  p.vcodes = a.v->codes;
  p.ksz = a.k->sz;
  p.vsz = a.v->sz;
  p.tile_mask = a.tile_mask;
  p.out = a.out;
  p.status = a.status;
  p.out_dtype = a.out_dtype;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.S = a.S; p.Tcap = a.k->Tcap;
  p.rep = a.Hq / a.Hkv;
  p.pairs = (p.rep + 1) / 2;
  p.nT = a.S / kT;
  p.causal = a.causal;
  p.lens = a.lens;
  p.wait_ns = a.pol.wait_ns;
  p.issue_limit = a.pol.issue_limit;
  p.codes_bytes = kvq_cache_codes_bytes(a.k);
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane_off[h] = a.layout.plane_off[h];
    p.bits[h] = a.layout.bits[h];
  }
  const float scale = a.softmax_scale > 0.0f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  const int64_t items = static_cast<int64_t>(p.nT) * a.B * a.Hkv * p.pairs;
  if (items >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  return D == 128 ? launch_prefill_d<128>(p, items, stream) : launch_prefill_d<64>(p, items, stream);
}

}  // namespace kvq
