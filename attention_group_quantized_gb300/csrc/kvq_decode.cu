// kvq_decode.cu -- decode attention over the group-quantised KV cache.
//
// Method: one query token per (sequence, query head) attends its sequence's
// cached keys; the cache holds integer codes with a per-group fp16 scale and
// zero point (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.4), and
// dequantisation happens inside the attention read (same page, §1.3).  The
// keys are visited tile by tile with an online softmax carrying the running
// max and normaliser (same page, §2.2); splits of the key range run on
// different CTAs and are merged by log-sum-exp.
//
// GB300 design (HBM-bound; the aim is few instructions per cache byte):
//  * Stream-K split: the (sequence, KV head, 64-token tile) work list is cut
//    into equal contiguous ranges, one per persistent CTA (SMs x CTAs/SM), so
//    ragged lengths cost no load imbalance; each CTA emits one partial
//    (o, lse) per segment piece it touched, and the CTA that completes a
//    segment (a per-segment arrival counter) merges its pieces in place -- no
//    second kernel.  A segment held by one CTA is written out directly.
//  * Eight warps in two warpgroups.  Warps 0-3 consume tiles, 16 tokens
//    each, two tiles of a piece per step for more independent work per
//    warp.  Warp 4 streams each tile's codes by TMA (2D tensor copies with
//    hardware swizzle) and its scale/zero words by 1D bulk copies into a
//    kStages-deep ring.  Warps 5 and 7 (even and odd tiles) turn the
//    scale/zero words of each landed tile into tables (fp32 scales carrying
//    the softmax scale, zero terms, tokens past the sequence end zeroed) so
//    the consumers do no per-group conversions.  Warp 6 runs piece ends
//    other than the CTA's last -- combining the consumers' states, writing
//    the partial, counting arrivals, merging -- while the consumers go on
//    with the next tiles; the last piece the consumers finish themselves.
//    setmaxnreg moves registers from the helper warpgroup to the consumers.
//  * The products run on the tensor cores with exact operands: a code byte
//    becomes the fp16 value 1024 + c by one byte permute.
//      S^T = K Q^T (rows = 16 tokens per warp, columns = the query heads of
//        the KV head), per group g of 32 channels: C_g = (1024 + c).Q, then
//        S += s_g C_g - (1024 + z_g) s_g sum_g(Q), which equals s_g (c - z_g).Q.
//        Each lane then holds two tokens of heads 2t, 2t+1 -- the same heads as
//        its output columns below, so the softmax factors need no shuffles.
//      O^T = V^T P^T (rows = channels, columns = query heads): each MMA's rows
//        lie in one group g, so its B operand is P^T * s_g (P rounded to fp16,
//        transposed in registers by movmatrix, times the fp16 scale); A is
//        1024 + c, and one extra MMA per group accumulates
//        sum_tok (1024 + z_g) P s_g into row g of a spare tile, subtracted at
//        the end.  Each such row must see the same MMAs with nonzero terms, in
//        the same order, as the output rows of its group (two spare tiles, even
//        and odd groups, keep that): the tensor core's fp32 accumulation then
//        rounds the large common 1024 * sum(P s_g) part the same way on both
//        sides and it cancels; a differently split sum leaves an error about
//        ten times larger.
//  * Fragments come from the swizzled code tiles by ldmatrix: K as stored
//    (token rows, a register holds four channels of one token), V transposed
//    (a register holds two tokens of two channels).  Every lane's row
//    addresses are fixed, and the swizzle keeps all eight rows of each 8x8
//    matrix in distinct banks.
//  * The cache is streamed with an L2 evict-first policy: it is read once per
//    call, and the small buffers the next call needs stay in L2.
//  * One CTA serves all query heads of a KV head, so every cache byte is read
//    once for the whole GQA group.
#include <cfloat>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_split.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kTile = 64;       // tokens per pipeline stage
constexpr int kWarps = 4;       // consumer warps; each owns 16 tokens of a tile
// two warpgroups: the consumers, then TMA issuer, table builder, epilogue and one idle warp
constexpr int kThreads = 2 * kWarps * 32;
// setmaxnreg split of the 128 registers a thread is launched with (tunable at build time)
#ifndef KVQ_DECODE_CONSUMER_REGS
#define KVQ_DECODE_CONSUMER_REGS 160
#endif
constexpr int kConsumerRegs = KVQ_DECODE_CONSUMER_REGS;
constexpr int kHelperRegs = 256 - kConsumerRegs;
static_assert(kWarps * (kConsumerRegs + kHelperRegs) == 2 * kWarps * 128, "register split must use the launch allocation");
// pipeline depth and CTAs per SM (tunable at build time)
#ifndef KVQ_DECODE_STAGES
#define KVQ_DECODE_STAGES 4
#endif
#ifndef KVQ_DECODE_MIN_BLOCKS
#define KVQ_DECODE_MIN_BLOCKS 2
#endif
// ring slots in shared memory; a call may keep fewer tiles in flight (its policy)
constexpr int kStages = KVQ_DECODE_STAGES;
constexpr int kMaxRep = 8;      // query heads per KV head
constexpr int kMaxL2Tiles = 16; // most tiles per CTA a policy may warm into L2

struct DParams {
  CUtensorMap tm_k8, tm_k4, tm_v8, tm_v4;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  const uint16_t* q;
  const int32_t* seq_lens;
  int32_t* ws_cnt;      // [B*Hkv] pieces written per segment; zero between calls
  float* ws_lse;        // [slots][rep]
  float* ws_o;          // [slots][rep][D]
  void* out;
  int32_t* status;
  int32_t out_dtype;
  int32_t B, Hq, Hkv, Tcap, rep, num_ctas;   // B sequences, Tcap tokens each at most
  // where a tile lives: without a block table, sequence b's tile i is row
  // (plane * pB + b) * pT + 64 i of the code planes (pB = B, pT = Tcap); with
  // one, it is page bt[b * bt_stride + i] of a pool of pB pages of pT = 64
  const int32_t* bt;
  int32_t bt_stride, pB, pT;
  float scale_log2;
  // per-call policy: tiles per CTA prefetched into L2 before the dependency
  // wait (0 .. kMaxL2Tiles), the bounded-wait limit, and the test-only issue
  // limit (tiles the copy issuer streams before it stops; negative = no
  // limit).  The ring depth (tiles kept in flight into shared memory) is the
  // kernel's template parameter RING.
  int32_t l2_warm, issue_limit;
  uint64_t wait_ns;
  int32_t plane[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

// Ring slot and phase parity of the k-th tile of a CTA's range in a ring of
// RING slots.  RING is 2 or 4: even, so each slot is only ever filled with
// even or only with odd tiles and one table warp waits on all of its phases.
template <int RING>
__device__ __forceinline__ void ring_pos(int k, int& slot, uint32_t& parity) {
  static_assert(RING == 2 || RING == 4, "ring depth 2 or 4");
  slot = k % RING;
  parity = static_cast<uint32_t>((k / RING) & 1);
}

// Hand-off buffer from the consumer warps to the epilogue warp at a piece end.
template <int D>
struct EpiBuf {
  float o[kWarps][kMaxRep][D];     // unnormalised output per consumer warp and head
  float ml[kWarps][kMaxRep][2];    // (running max, sum) per consumer warp and head, log2 domain
  int4 info;                       // sequence, KV head
  int flag[2];                     // last-arrival flags: epilogue warp, consumer warps
};

template <int D>
struct Smem {
  static constexpr int G = D / 32;
  static constexpr int kCodeBytes = kTile * D;          // room for an 8-bit tile
  static constexpr int kSzBytes = kTile * G * 4;
  // offsets inside a stage
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kCodeBytes;
  static constexpr int kOffKsz = 2 * kCodeBytes;          // raw K scale/zero words [64 tok][G] ...
  static constexpr int kOffVsz = kOffKsz + kSzBytes;       // ... and V's, both replaced by
  // K table, float4 [G][4 warps][8 rows r]: (s, (1024 + z) s) of tokens 16w + r
  // and 16w + r + 8, the scale carrying the softmax scale
  static constexpr int kOffKt = kOffKsz;
  // V tables, uint2 [G][4 warps][4 columns c]: half2 pairs of tokens
  // (16w + 2c, 16w + 2c + 1) and (16w + 8 + 2c, 16w + 9 + 2c): s, and (1024 + z)
  static constexpr int kOffVtS = kOffKt + kTile * G * 8;
  static constexpr int kOffVtZ = kOffVtS + kTile * G * 2;
  static constexpr int kOffMeta = kOffVtZ + kTile * G * 2; // int4 {b, kvh, i | flags, len}
  static constexpr int kOffQ = kOffMeta + 16;              // bf16 [rep][D]: the piece's queries (first tile)
  static constexpr int kStageBytes = ((kOffQ + kMaxRep * D * 2 + 1023) / 1024) * 1024;
  static_assert(kOffKt + kTile * G * 8 == kOffVsz + kSzBytes, "the K table exactly covers the raw words");
  static constexpr int kOffEpi = kStages * kStageBytes;                       // EpiBuf<D>
  static constexpr int kOffBars = kOffEpi + ((static_cast<int>(sizeof(EpiBuf<D>)) + 15) / 16) * 16;
  static constexpr int kBars = (3 * kStages + 3) * 8;
  static constexpr int kFixed = kOffBars + kBars;
  static size_t bytes(int B) { return 1024 + kFixed + static_cast<size_t>(B + 1) * 4 * 2; }
};

// tile flags (meta.z): tile index in bits 0-23, then
constexpr int kFlag4 = 1 << 24;      // the KV head is stored with 4-bit codes
constexpr int kFlagFull = 1 << 25;   // every token of the tile is inside the sequence
constexpr int kFlagEnd = 1 << 29;    // last tile of a piece
constexpr int kFlagStart = 1 << 30;  // first tile of a piece

// Byte offset of (row, byte) inside a TMA tile written with the swizzle mode
// matching its row pitch R (128B, 64B or 32B): the 16-byte chunk index is
// XORed with address bits 7.. of the row start.
template <int R>
__device__ __forceinline__ uint32_t swz(int row, int byte) {
  if constexpr (R == 128) return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
  if constexpr (R == 64) return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15));
  return row * 32 + ((((byte >> 4) ^ ((row >> 2) & 1)) << 4) | (byte & 15));
}

// (d0, d1) += (a, a) * (b0, b1) as one two-wide fp32 instruction
__device__ __forceinline__ void ffma2_b(float& d0, float& d1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %2};\n\t"
      "mov.b64 rb, {%3, %4};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a), "f"(b0), "f"(b1));
}

using split::Cursor;
using split::advance;
using split::locate;
using split::count_pieces;

// Per-thread shared-memory offsets (from a stage base) of the ldmatrix rows this
// lane supplies; they do not change from tile to tile.  m = l >> 3 is the
// matrix the lane addresses.
//   K (as stored):  token row 16w + 8(m & 1) + (l & 7), chunk (m >> 1)
//   V (transposed): token row 16w + 8(m >> 1) + (l & 7), chunk (m & 1)
struct LaneAddr {
  uint32_t k8, k4, v8, v4;
};

// Other chunks of the same row differ only by an XOR of the swizzled offset:
// two chunks further flips address bit 5, one group of V codes further too.
template <int D>
__device__ __forceinline__ LaneAddr lane_addr(int w, int lane) {
  constexpr int R8 = D, R4 = D / 2;
  LaneAddr a;
  const int m = lane >> 3;
  const int r = 16 * w + 8 * (m & 1) + (lane & 7);
  a.k8 = swz<R8>(r, 16 * (m >> 1));
  a.k4 = swz<R4>(r, 16 * (m >> 1));
  const int vr = 16 * w + 8 * (m >> 1) + (lane & 7);
  a.v8 = swz<R8>(vr, 16 * (m & 1));
  a.v4 = swz<R4>(vr, 16 * (m & 1));
  return a;
}

// Q fragments of S^T = K Q^T (B operand columns = the group's query heads,
// zero from rep up) in the channel order of the code unpacking, and per-group
// sums of the same fp16 values for head g (reduced over the quad).
//   8-bit: k-step s (16 channels): cols 2t,2t+1 <-> ch 16s + 4t + {0,1},
//          cols 2t+8, 2t+9 <-> ch 16s + 4t + {2,3}
//   4-bit: k-steps 2g, 2g+1 of group g: ch 32g + 8t + {(0,4),(1,5)} and {(2,6),(3,7)}
template <int D>
__device__ __forceinline__ void load_q(uint32_t (&qa)[D / 16][2], float (&qsum)[D / 32], const DParams& p,
                                       const uint16_t* qs, int bits, int g, int t) {
  constexpr int G = D / 32;
  const uint16_t* src = qs + g * D;
  bool ok = true;
#pragma unroll
  for (int grp = 0; grp < G; ++grp) {
    float f[8];   // 8-bit: ch 32grp + {4t..4t+3, 16+4t..16+4t+3}; 4-bit: ch 32grp + 8t + 0..7
    if (g < p.rep) {
      uint32_t w[4];
      if (bits == 8) {
        const uint2 a = *reinterpret_cast<const uint2*>(src + grp * 32 + 4 * t);
        const uint2 c = *reinterpret_cast<const uint2*>(src + grp * 32 + 16 + 4 * t);
        w[0] = a.x; w[1] = a.y; w[2] = c.x; w[3] = c.y;
      } else {
        const uint4 a = *reinterpret_cast<const uint4*>(src + grp * 32 + 8 * t);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ok &= fabsf(f[i]) < 65504.0f;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.0f;
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += __half2float(__float2half_rn(f[i]));
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    qsum[grp] = s;
    if (bits == 8) {
      qa[2 * grp][0] = pack_half2(f[0], f[1]);
      qa[2 * grp][1] = pack_half2(f[2], f[3]);
      qa[2 * grp + 1][0] = pack_half2(f[4], f[5]);
      qa[2 * grp + 1][1] = pack_half2(f[6], f[7]);
    } else {
      qa[2 * grp][0] = pack_half2(f[0], f[4]);
      qa[2 * grp][1] = pack_half2(f[1], f[5]);
      qa[2 * grp + 1][0] = pack_half2(f[2], f[6]);
      qa[2 * grp + 1][1] = pack_half2(f[3], f[7]);
    }
  }
  if (!ok) report(p.status, KVQ_ERR_NONFINITE);
}

// Scores of the warp's 16 tokens: S^T = K Q^T with the tokens as the MMA rows
// and the query heads as its columns, so S[0], S[1] are token 16w + g with
// heads 2t, 2t+1 and S[2], S[3] token 16w + g + 8.  The A operand comes by
// ldmatrix from the swizzled code tile (a register holds four channels of one
// token); per group the product is rescaled with the tile's K table:
// S += s C_g - (1024 + z) s sum_g(q).
template <int D, int BITS>
__device__ __forceinline__ void qk_tile(float (&S)[4], const uint32_t (&qa)[D / 16][2], const float (&qs)[D / 32][2],
                                        uint32_t st_s, const uint8_t* st, const LaneAddr& la, int w, int g) {
  using L = Smem<D>;
  constexpr int G = D / 32;
  const float4* kt = reinterpret_cast<const float4*>(st + L::kOffKt) + w * 8 + g;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  // one ldmatrix: tokens 0-7 and 8-15 of two chunks; 8-bit: the two chunks of
  // group pr, 4-bit: groups 2pr and 2pr + 1
#pragma unroll
  for (int pr = 0; pr < (BITS == 8 ? G : (G + 1) / 2); ++pr) {
    uint32_t r[4];
    if constexpr (BITS == 8) {
      ldsm_x4(r, st_s + L::kOffK + (la.k8 ^ (static_cast<uint32_t>(pr) << 5)));
    } else {
      ldsm_x4(r, st_s + L::kOffK + (la.k4 ^ (static_cast<uint32_t>(pr) << 5)));
    }
#pragma unroll
    for (int gg = 0; gg < (BITS == 8 ? 1 : 2); ++gg) {
      const int grp = BITS == 8 ? pr : 2 * pr + gg;
      float c[4];
      if constexpr (BITS == 8) {
        mma_16816_z(c, bytes01_biased(r[0]), bytes01_biased(r[1]), bytes23_biased(r[0]), bytes23_biased(r[1]),
                    qa[2 * grp][0], qa[2 * grp][1]);
        mma_16816(c, bytes01_biased(r[2]), bytes01_biased(r[3]), bytes23_biased(r[2]), bytes23_biased(r[3]),
                  qa[2 * grp + 1][0], qa[2 * grp + 1][1]);
      } else {
        const uint32_t w0 = r[2 * gg], w1 = r[2 * gg + 1];
        const uint32_t w08 = w0 >> 8, w18 = w1 >> 8;
        mma_16816_z(c, nib_biased(w0), nib_biased(w1), nib_hi_biased(w0), nib_hi_biased(w1), qa[2 * grp][0],
                    qa[2 * grp][1]);
        mma_16816(c, nib_biased(w08), nib_biased(w18), nib_hi_biased(w08), nib_hi_biased(w18),
                  qa[2 * grp + 1][0], qa[2 * grp + 1][1]);
      }
      const float4 sz = kt[grp * 32];   // tokens g and g + 8
      // the lane's two heads at once (same rounding as two scalar FMAs)
      ffma2_b(acc[0], acc[1], -sz.y, qs[grp][0], qs[grp][1]);
      ffma2_b(acc[0], acc[1], sz.x, c[0], c[1]);
      ffma2_b(acc[2], acc[3], -sz.w, qs[grp][0], qs[grp][1]);
      ffma2_b(acc[2], acc[3], sz.z, c[2], c[3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) S[i] = acc[i];
}

// O^T[ch][h] += (1024 + c)[ch][tok] (P s_g)[tok][h] over the warp's 16 tokens,
// and Z[g & 1][g][h] += (1024 + z_g)[tok] (P s_g)[tok][h] in row g of a spare
// tile (two accumulators, even and odd groups: each row sees the same MMAs
// with nonzero terms, in the same order, as the output rows of its group).
// pb = P^T as the B operand: tokens 2t, 2t+1 | 8+2t, 9+2t of head g, fp16.
// A operand (rows = channels, k = tokens) by transposed ldmatrix from the
// swizzled code tile.  Row -> channel of m-tile 2*grp + mh:
//   8-bit: row r < 8 -> 32grp + 2r + mh, row r >= 8 -> 32grp + 16 + 2(r-8) + mh
//   4-bit: row r < 8 -> 32grp + 4r + 2mh, row r >= 8 -> 32grp + 4(r-8) + 2mh + 1
// Accumulators hold heads 2t (c0, c2) and 2t+1 (c1, c3).
template <int D, int BITS>
__device__ __forceinline__ void pv_tile(float (&O)[D / 16][4], float (&Z)[2][4], const uint32_t (&pb)[2],
                                        uint32_t st_s, const uint8_t* st, const LaneAddr& la, int w, int g,
                                        int t) {
  using L = Smem<D>;
  constexpr int G = D / 32;
  const uint2* vts = reinterpret_cast<const uint2*>(st + L::kOffVtS) + w * 4 + t;
  // row g of the zero-term product carries group g: lanes with g < G load it once
  uint2 zown = make_uint2(0u, 0u);
  if (g < G) zown = reinterpret_cast<const uint2*>(st + L::kOffVtZ)[(g * 4 + w) * 4 + t];
  uint32_t rv4[2][4];
  if constexpr (BITS == 4) {
    ldsm_x4_t(rv4[0], st_s + L::kOffV + la.v4);
    if constexpr (G == 4) ldsm_x4_t(rv4[1], st_s + L::kOffV + (la.v4 ^ 32u));
  }
#pragma unroll
  for (int grp = 0; grp < G; ++grp) {
    const uint2 sv = vts[grp * 16];   // s_g of tokens 2t, 2t+1 | 8+2t, 9+2t
    const uint32_t b0 = hmul2_u32(pb[0], sv.x);
    const uint32_t b1 = hmul2_u32(pb[1], sv.y);
    if constexpr (BITS == 8) {
      uint32_t r[4];   // (tok 0-7, ch 0-15), (tok 0-7, ch 16-31), (tok 8-15, ch 0-15), (tok 8-15, ch 16-31)
      ldsm_x4_t(r, st_s + L::kOffV + (la.v8 ^ (static_cast<uint32_t>(grp) << 5)));
      mma_16816(O[2 * grp + 0], bytes02_biased(r[0]), bytes02_biased(r[1]), bytes02_biased(r[2]),
                bytes02_biased(r[3]), b0, b1);
      mma_16816(O[2 * grp + 1], bytes13_biased(r[0]), bytes13_biased(r[1]), bytes13_biased(r[2]),
                bytes13_biased(r[3]), b0, b1);
    } else {
      // matrices of ldmatrix (gi = grp/2): (group 2gi, tok 0-7), (2gi+1, 0-7), (2gi, 8-15), (2gi+1, 8-15)
      const uint32_t lo = rv4[grp >> 1][grp & 1], hi = rv4[grp >> 1][2 + (grp & 1)];
      const uint32_t lo8 = lo >> 8, hi8 = hi >> 8;
      mma_16816(O[2 * grp + 0], nib_biased(lo), nib_hi_biased(lo), nib_biased(hi), nib_hi_biased(hi), b0, b1);
      mma_16816(O[2 * grp + 1], nib_biased(lo8), nib_hi_biased(lo8), nib_biased(hi8), nib_hi_biased(hi8), b0, b1);
    }
    const uint32_t za = g == grp ? zown.x : 0u;
    const uint32_t zb = g == grp ? zown.y : 0u;
    mma_16816(Z[grp & 1], za, 0u, zb, 0u, b0, b1);
  }
}

// channel held by accumulator row half (0: rows < 8, 1: rows >= 8) of m-tile (grp, mh), thread row g
template <int BITS>
__device__ __forceinline__ int acc_channel(int grp, int mh, int half, int g) {
  if constexpr (BITS == 8) return 32 * grp + 16 * half + 2 * g + mh;
  return 32 * grp + 4 * g + 2 * mh + half;
}

// Sequences of length 0 get a zero output row (no CTA visits them); one warp
// per CTA writes its share of the rows.
template <int D>
__device__ __forceinline__ void zero_empty_rows(const DParams& p, const int32_t* lens, int lane) {
  const int n = p.B * p.Hq * D;
  for (int idx = blockIdx.x * 32 + lane; idx < n; idx += gridDim.x * 32) {
    const int b = idx / (p.Hq * D);
    if (lens[b] == 0) {
      if (p.out_dtype == KVQ_OUT_F32) reinterpret_cast<float*>(p.out)[idx] = 0.0f;
      else reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(0.0f);
    }
  }
}

// The G scale/zero words of one token (16 or 8 bytes, aligned).
template <int G>
__device__ __forceinline__ void load_words(uint32_t (&w)[G], const uint32_t* src) {
  if constexpr (G == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    w[0] = v.x; w[1] = v.y;
  }
}

template <int D>
__device__ __forceinline__ void store_out4(const DParams& p, int64_t i, float4 v) {
  if (!KVQ_IN_RANGE(i >= 0 && i + 4 <= static_cast<int64_t>(p.B) * p.Hq * D, p.status)) return;
  if (p.out_dtype == KVQ_OUT_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + i) = v;
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + i) = u;
  }
}

// Thread-group synchronisation for segment_end: the epilogue warp uses
// __syncwarp; the four consumer warps a bounded mbarrier round (a plain
// bar.sync could wait forever if one warp left after a timed-out wait).
struct WarpSync {
  __device__ __forceinline__ void operator()() const { __syncwarp(); }
};
struct ConsumerSync {
  uint64_t* bar;
  uint32_t* phase;
  bool* ok;
  int32_t* status;
  uint64_t wait_ns;
  __device__ __forceinline__ void operator()() const {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    *ok = *ok && mbar_wait(bar, *phase & 1, status, wait_ns);
    ++*phase;
    __syncwarp();
  }
};

// End of a piece.  The four consumer warps' states (running max and sum per
// head, unnormalised o per head and channel) sit in the hand-off buffer.  A
// segment held by this CTA alone is normalised and written out; otherwise the
// CTA's partial (o, lse) goes to the workspace and the CTA whose arrival
// completes the segment merges all its pieces by log-sum-exp.  Run by
// `nthr` threads (tid = 0 .. nthr-1) that `sync` joins; `epi_empty`, if
// given, is arrived once the buffer has been read.
template <int D, int MB, class Sync>
__device__ __forceinline__ void segment_end(const DParams& p, const EpiBuf<D>* eb, int* flag, int cb, int ckvh,
                                            const int32_t* pre, int64_t N, int C, int tid, int nthr,
                                            const Sync& sync, uint64_t* epi_empty) {
  const int Hkv = p.Hkv, rep = p.rep;
  const int seg = cb * Hkv + ckvh;
  int c0, c1;   // CTAs holding the first and the last tile of the segment
  split::segment_ctas(pre, Hkv, cb, ckvh, N, C, &c0, &c1);
  const bool whole = c0 == c1;
  const int64_t orow0 = (static_cast<int64_t>(cb) * p.Hq + ckvh * rep) * D;
  const int64_t slot = static_cast<int64_t>(seg) + blockIdx.x;
  // debug build: the segment's counter and this piece's workspace slot exist
  // (slots = segments + split CTAs); a failed check writes no partial
  const int64_t n_slots = static_cast<int64_t>(p.B) * Hkv + p.num_ctas;
  const bool slot_ok = KVQ_IN_RANGE(seg < p.B * Hkv && slot < n_slots && c1 < p.num_ctas, p.status);
  for (int i4 = tid; i4 < rep * (D / 4); i4 += nthr) {
    const int h = i4 / (D / 4), ch = (i4 % (D / 4)) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, eb->ml[ww][h][0]);
    float Lsum = 0.0f;
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (M != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float sc = fast_exp2(eb->ml[ww][h][0] - M);
        Lsum += eb->ml[ww][h][1] * sc;
        const float4 v = *reinterpret_cast<const float4*>(&eb->o[ww][h][ch]);
        o.x += v.x * sc; o.y += v.y * sc; o.z += v.z * sc; o.w += v.w * sc;
      }
    }
    const bool any = M != -INFINITY && Lsum > 0.0f;
    const float inv = any ? 1.0f / Lsum : 0.0f;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
    if (whole) {
      store_out4<D>(p, orow0 + static_cast<int64_t>(h) * D + ch, o);
    } else if (slot_ok) {
      *reinterpret_cast<float4*>(p.ws_o + (slot * rep + h) * D + ch) = o;
      if (ch == 0) p.ws_lse[slot * rep + h] = any ? M + __log2f(Lsum) : -INFINITY;
    }
  }
  if (epi_empty != nullptr || !whole) sync();   // the group's reads of eb / stores are done
  if (epi_empty != nullptr && tid == 0) mbar_arrive(epi_empty);   // the consumers may refill the buffer
  if (whole) return;
  // publish the piece and count the arrivals with one acquire-release
  // atomic: after the group barrier its release orders every member's partial
  // stores (release is cumulative) before the count, and for the last
  // arriver its acquire orders the other pieces' stores, released by their
  // own arrivals, before the group's reads below
  if (tid == 0) {
    const int np = c1 - c0 + 1;   // every split CTA owns at least one tile
    *flag = (slot_ok && atom_add_acq_rel_gpu(p.ws_cnt + seg, 1) + 1 == np) ? 1 : 0;
  }
  sync();
  if (*flag != 1) return;
  // the segment is complete: log-sum-exp over its pieces, four channels per
  // thread, MB pieces per round with all their loads in flight together
  for (int i4 = tid; i4 < rep * (D / 4); i4 += nthr) {
    const int h = i4 / (D / 4), ch = (i4 % (D / 4)) * 4;
    float M = -INFINITY, Lsum = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int cb4 = c0; cb4 <= c1; cb4 += MB) {
      float lse[MB];
      float4 v[MB];
#pragma unroll
      for (int u = 0; u < MB; ++u) {
        const int c = cb4 + u;
        const bool live = c <= c1;
        const int64_t sl = static_cast<int64_t>(seg) + (live ? c : c0);
        lse[u] = live ? __ldcg(p.ws_lse + sl * rep + h) : -INFINITY;
        v[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (sl * rep + h) * D + ch));
      }
      float Mr = M;
#pragma unroll
      for (int u = 0; u < MB; ++u) Mr = fmaxf(Mr, lse[u]);
      if (Mr == -INFINITY) continue;   // no piece with weight yet
      const float a = M == -INFINITY ? 0.0f : fast_exp2(M - Mr);
      acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
      Lsum *= a;
#pragma unroll
      for (int u = 0; u < MB; ++u) {
        const float bw = lse[u] == -INFINITY ? 0.0f : fast_exp2(lse[u] - Mr);
        acc.x += bw * v[u].x; acc.y += bw * v[u].y; acc.z += bw * v[u].z; acc.w += bw * v[u].w;
        Lsum += bw;
      }
      M = Mr;
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    store_out4<D>(p, orow0 + static_cast<int64_t>(h) * D + ch, acc);
  }
  if (tid == 0) p.ws_cnt[seg] = 0;   // ready for the next call
}

// One consumer step over NT tiles (1, or 2 of the same piece) for the warp's
// 16 tokens of each: scores, one online-softmax update over all of them, and
// the P.V products.  lim[u] = tokens of tile u inside the sequence.  The
// running max m_run and the per-lane partial sums l_run are those of heads
// 2t, 2t+1 -- the same heads as the lane's output accumulator columns.
template <int D, int BITS, int NT>
__device__ __forceinline__ void consume_tiles(const uint32_t (&st_s)[NT], const uint8_t* const (&st)[NT],
                                              const int (&lim)[NT], const uint32_t (&qa)[D / 16][2],
                                              const float (&qs)[D / 32][2], float (&O)[D / 16][4],
                                              float (&Z)[2][4], float (&m_run)[2], float (&l_run)[2],
                                              const LaneAddr& la, int w, int g, int t) {
  float S[NT][4];   // log2-domain scores (the table carries the softmax scale)
#pragma unroll
  for (int u = 0; u < NT; ++u) qk_tile<D, BITS>(S[u], qa, qs, st_s[u], st[u], la, w, g);
  // mask past the sequence end (only the last tile of a sequence)
  const int r0 = 16 * w + g;
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    if (r0 >= lim[u]) S[u][0] = S[u][1] = -INFINITY;
    if (r0 + 8 >= lim[u]) S[u][2] = S[u][3] = -INFINITY;
  }
  // online softmax for heads 2t, 2t+1: the max over the warp's tokens (rows g).
  // While no score exceeds the running max the max is unchanged and so is
  // every factor: the warp reduction and the rescale run only when some lane
  // sees a larger score (the results are the same either way).
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    mx0 = fmaxf(mx0, fmaxf(S[u][0], S[u][2]));
    mx1 = fmaxf(mx1, fmaxf(S[u][1], S[u][3]));
  }
  float a0 = 1.0f, a1 = 1.0f;
  if (__any_sync(0xffffffffu, mx0 > m_run[0] || mx1 > m_run[1])) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    a0 = fast_exp2(m_run[0] - (mn0 == -INFINITY ? 0.0f : mn0));
    a1 = fast_exp2(m_run[1] - (mn1 == -INFINITY ? 0.0f : mn1));
    m_run[0] = mn0;
    m_run[1] = mn1;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      O[i][0] *= a0; O[i][1] *= a1;
      O[i][2] *= a0; O[i][3] *= a1;
    }
#pragma unroll
    for (int z = 0; z < 2; ++z) {
      Z[z][0] *= a0; Z[z][1] *= a1; Z[z][2] *= a0; Z[z][3] *= a1;
    }
  }
  const float mu0 = m_run[0] == -INFINITY ? 0.0f : m_run[0];
  const float mu1 = m_run[1] == -INFINITY ? 0.0f : m_run[1];
  float P[NT][4];
  float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    P[u][0] = fast_exp2(S[u][0] - mu0);
    P[u][1] = fast_exp2(S[u][1] - mu1);
    P[u][2] = fast_exp2(S[u][2] - mu0);
    P[u][3] = fast_exp2(S[u][3] - mu1);
    ps0 += P[u][0] + P[u][2];
    ps1 += P[u][1] + P[u][3];
  }
  l_run[0] = l_run[0] * a0 + ps0;
  l_run[1] = l_run[1] * a1 + ps1;
  // P^T as the B operand of the products: transpose the (token, head) pairs
  // of tokens g and g + 8 into (head g; tokens 2t, 2t+1) and (8+2t, 9+2t)
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    const uint32_t pb[2] = {movm_trans(pack_half2(P[u][0], P[u][1])), movm_trans(pack_half2(P[u][2], P[u][3]))};
    pv_tile<D, BITS>(O, Z, pb, st_s[u], st[u], la, w, g, t);
  }
}

// Before the dependency wait (one warp): prefetch into L2 the first p.l2_warm
// tiles of this CTA's range, so that the copies issued after the wait find
// them there while the previous kernel's last CTAs still run.  The lengths
// read here may be stale -- the previous kernel may still be writing them --
// but they only choose which lines to prefetch (clamped into the cache), and
// an L2 prefetch returns nothing to the program, so no result depends on
// them.  Batches of more than 32 sequences skip the warm-up.
template <int D, bool PAGED>
__device__ __forceinline__ void warm_l2(const DParams& p, int lane) {
  constexpr int G = D / 32;
  if (p.l2_warm <= 0 || p.B > 32) return;
  int len = lane < p.B ? p.seq_lens[lane] : 0;
  len = min(max(len, 0), p.Tcap);
  const int n = (len + kTile - 1) / kTile;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const int64_t N = static_cast<int64_t>(p.Hkv) * total;
  const int C = N < p.num_ctas ? static_cast<int>(N) : p.num_ctas;
  if (N == 0 || static_cast<int>(blockIdx.x) >= C) return;
  const int64_t f0 = N * blockIdx.x / C, f1 = N * (blockIdx.x + 1) / C;
  const int64_t f = f0 + lane;   // this lane's tile
  // its sequence: the number of sequences ending at or before f
  int b = 0;
  for (int s = 0; s < p.B; ++s) b += static_cast<int64_t>(p.Hkv) * __shfl_sync(0xffffffffu, incl, s) <= f ? 1 : 0;
  const int bs = min(b, p.B - 1);
  const int nb = __shfl_sync(0xffffffffu, n, bs);
  const int eb = __shfl_sync(0xffffffffu, incl, bs) - nb;
  if (lane >= p.l2_warm || f >= f1 || b >= p.B || nb == 0) return;
  const int64_t off = f - static_cast<int64_t>(p.Hkv) * eb;
  const int kvh = static_cast<int>(off / nb), i = static_cast<int>(off % nb);
  const int bits = p.bits[kvh];
  int pb = bs, pt = i * kTile;
  if constexpr (PAGED) {   // (a stale or bad page id only misdirects this prefetch)
    if (!KVQ_IN_RANGE(i < p.bt_stride, p.status)) return;
    pb = min(max(p.bt[static_cast<int64_t>(bs) * p.bt_stride + i], 0), p.pB - 1);
    pt = 0;
  }
  const int32_t row0 = (p.plane[kvh] * p.pB + pb) * p.pT + pt;
  const int64_t szoff = (static_cast<int64_t>(kvh) * p.pB + pb) * p.pT + pt;
  if (!KVQ_IN_RANGE(kvh < p.Hkv && szoff + kTile <= static_cast<int64_t>(p.Hkv) * p.pB * p.pT, p.status)) return;
  prefetch_l2_tile_2d(bits == 8 ? &p.tm_k8 : &p.tm_k4, 0, row0);
  prefetch_l2_tile_2d(bits == 8 ? &p.tm_v8 : &p.tm_v4, 0, row0);
  prefetch_l2_bulk(p.k_sz + szoff * G, Smem<D>::kSzBytes);
  prefetch_l2_bulk(p.v_sz + szoff * G, Smem<D>::kSzBytes);
}

// PAGED: the tiles are pages of a pool found through p.bt (a separate
// instantiation, so the contiguous kernel carries none of it).  RING: tiles
// kept in flight into shared memory (the policy's ring depth, 2 or kStages).
template <int D, bool PAGED, int RING>
__global__ void __launch_bounds__(kThreads, KVQ_DECODE_MIN_BLOCKS) decode_split_kernel(const __grid_constant__ DParams p) {
  using L = Smem<D>;
  constexpr int G = D / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  EpiBuf<D>* eb = reinterpret_cast<EpiBuf<D>*>(smem + L::kOffEpi);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
  uint64_t* ready = full + kStages;
  uint64_t* empty = ready + kStages;
  uint64_t* epi_full = empty + kStages;    // consumers -> epilogue: a piece's states are in eb
  uint64_t* epi_empty = epi_full + 1;      // epilogue -> consumers: eb may be overwritten
  uint64_t* gbar = epi_empty + 1;          // consumer-group barrier for the final piece
  int32_t* pre = reinterpret_cast<int32_t*>(smem + L::kFixed);
  int32_t* lens = pre + (p.B + 1);

  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int B = p.B, Hkv = p.Hkv;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(epi_full, kWarps);
    mbar_init(epi_empty, 1);
    mbar_init(gbar, kWarps);
    fence_barrier_init();
  }
  if (tid == kWarps * 32) {
    prefetch_tmap(&p.tm_k8);
    prefetch_tmap(&p.tm_v8);
    prefetch_tmap(&p.tm_k4);
    prefetch_tmap(&p.tm_v4);
  }
  if (w == kWarps) warm_l2<D, PAGED>(p, lane);
  // With programmatic dependent launch this kernel may start while the
  // previous kernel in the stream is finishing: wait for it (and its memory)
  // before the first global access whose data is used, then let the next one
  // start early.
  grid_dependency_wait();
  grid_launch_dependents();
  // The lengths, clamped into the cache, and per-sequence tile counts with
  // their prefix sums.  Up to 32 sequences, warp 0 alone loads and scans them
  // (one block barrier after the wait); more are loaded by all threads first.
  auto load_len = [&](int b) {
    int L0 = p.seq_lens[b];
    if (L0 < 0 || L0 > p.Tcap) {
      report(p.status, KVQ_ERR_INVALID_ARG);
      L0 = L0 < 0 ? 0 : p.Tcap;
    }
    return L0;
  };
  const bool small_b = B <= 32;
  if (!small_b) {
    for (int b = tid; b < B; b += blockDim.x) lens[b] = load_len(b);
    __syncthreads();
  }
  if (w == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int len = 0;
      if (b < B) {
        len = small_b ? load_len(b) : lens[b];
        if (small_b) lens[b] = len;
      }
      int n = (len + kTile - 1) / kTile;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, n, o);
        if (lane >= o) n += v;
      }
      if (b < B) pre[b + 1] = carry + n;
      carry += __shfl_sync(0xffffffffu, n, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  __syncthreads();

  const int64_t N = static_cast<int64_t>(Hkv) * pre[B];
  // never more split CTAs than tiles: every CTA of the split then owns at
  // least one tile, and a segment's pieces are those of CTAs c0 .. c1
  const int C = N < p.num_ctas ? static_cast<int>(N) : p.num_ctas;
  const bool in_split = static_cast<int>(blockIdx.x) < C;
  // N c / C in 32 bits when the product fits (a 64-bit division is a long
  // software sequence on this critical path)
  auto cut = [&](int c) -> int64_t {
    const int64_t nc = N * c;
    return nc <= 0xFFFFFFFFll ? static_cast<int64_t>(static_cast<uint32_t>(nc) / static_cast<uint32_t>(C)) : nc / C;
  };
  const int64_t f0 = in_split ? cut(blockIdx.x) : 0;
  const int64_t f1 = in_split ? cut(blockIdx.x + 1) : 0;
  const int ntiles = static_cast<int>(f1 - f0);
  if (ntiles <= 0) {
    if (w == 0) zero_empty_rows<D>(p, lens, lane);
    return;
  }

  // Registers: launched with 128 per thread (checked on the host); the
  // consumer warpgroup takes kConsumerRegs, the helper warpgroup keeps
  // kHelperRegs: 4 x (kConsumerRegs + kHelperRegs) = 8 x 128, and per
  // sub-partition 32 x (kConsumerRegs + kHelperRegs) x 2 CTAs = 16384, its
  // whole register file.
  if (w >= kWarps) {
    tc::reg_dealloc<kHelperRegs>();
    if (w == kWarps) {
      // ---------------- TMA issuer warp: lane 0 keeps RING tiles in flight ----------------
      if (lane != 0) return;
      const uint64_t pol = l2_evict_first_policy();   // the cache is streamed once per call
      Cursor pc = locate(f0, pre, B, Hkv);
      // paged caches: the page ids are loaded kStages tiles ahead of their
      // copies (a ring of registers), so the lookups overlap the stage waits
      Cursor pa = pc;
      int pg[kStages];
#pragma unroll
      for (int j = 0; j < kStages; ++j) {
        pg[j] = 0;
        if (PAGED && j < ntiles) {
          pg[j] = KVQ_IN_RANGE(pa.b < p.B && pa.i < p.bt_stride, p.status)
                      ? p.bt[static_cast<int64_t>(pa.b) * p.bt_stride + pa.i] : 0;
          advance(pa, pre, B, Hkv);
        }
      }
      // test-only: the policy's issue limit stops streaming early (a bound
      // on the loop, so the per-tile code is the same either way)
      const int n_issue = p.issue_limit >= 0 && p.issue_limit < ntiles ? p.issue_limit : ntiles;
      for (int k = 0; k < n_issue; ++k) {
        int slot;
        uint32_t par;
        ring_pos<RING>(k, slot, par);
        if (k >= RING && !mbar_wait(&empty[slot], par ^ 1u, p.status, p.wait_ns)) return;
        uint8_t* st = smem + slot * L::kStageBytes;
        const int bits = p.bits[pc.kvh];
        const int Rb = D * bits / 8;
        int pb = pc.b, pt = pc.i * kTile;
        if constexpr (PAGED) {
          pb = pg[0];
#pragma unroll
          for (int j = 0; j + 1 < kStages; ++j) pg[j] = pg[j + 1];
          pg[kStages - 1] = 0;
          if (k + kStages < ntiles) {
            pg[kStages - 1] = KVQ_IN_RANGE(pa.b < p.B && pa.i < p.bt_stride, p.status)
                                  ? p.bt[static_cast<int64_t>(pa.b) * p.bt_stride + pa.i] : 0;
            advance(pa, pre, B, Hkv);
          }
          if (pb < 0 || pb >= p.pB) {   // a page outside the pool: report, read page 0 instead
            report(p.status, KVQ_ERR_INVALID_ARG);
            pb = 0;
          }
          pt = 0;
        }
        const int32_t row0 = (p.plane[pc.kvh] * p.pB + pb) * p.pT + pt;
        int64_t szoff = (static_cast<int64_t>(pc.kvh) * p.pB + pb) * p.pT + pt;
        // debug build: the tile's rows inside its code plane, its scale/zero
        // words and queries inside their buffers (a failed check reads the
        // buffers' first entries instead)
        (void)KVQ_IN_RANGE(row0 >= 0 && row0 + kTile <= (p.plane[pc.kvh] + 1) * p.pB * p.pT, p.status);
        if (!KVQ_IN_RANGE(szoff >= 0 && szoff + kTile <= static_cast<int64_t>(p.Hkv) * p.pB * p.pT, p.status))
          szoff = 0;
        uint64_t* bar = &full[slot];
        const bool first = pc.i == 0 || k == 0;
        const uint32_t qbytes = first ? static_cast<uint32_t>(p.rep * D * 2) : 0u;
        int64_t qoff = (static_cast<int64_t>(pc.b) * p.Hq + pc.kvh * p.rep) * D;
        if (!KVQ_IN_RANGE(qoff >= 0 && qoff + p.rep * D <= static_cast<int64_t>(p.B) * p.Hq * D, p.status)) qoff = 0;
        mbar_arrive_expect_tx(bar, 2 * kTile * Rb + 2 * L::kSzBytes + qbytes);
        if (first)
          bulk_g2s(st + L::kOffQ, p.q + qoff, qbytes, bar);
        tma_2d_g2s_hint(st + L::kOffK, bits == 8 ? &p.tm_k8 : &p.tm_k4, 0, row0, bar, pol);
        tma_2d_g2s_hint(st + L::kOffV, bits == 8 ? &p.tm_v8 : &p.tm_v4, 0, row0, bar, pol);
        bulk_g2s_hint(st + L::kOffKsz, p.k_sz + szoff * G, L::kSzBytes, bar, pol);
        bulk_g2s_hint(st + L::kOffVsz, p.v_sz + szoff * G, L::kSzBytes, bar, pol);
        advance(pc, pre, B, Hkv);
      }
      return;
    }
    if (w == kWarps + 1 || w == kWarps + 3) {
      // ---------------- two table warps (even / odd tiles): scale/zero words -> consumer tables ----------------
      const int par = w == kWarps + 1 ? 0 : 1;
      if (par >= ntiles) return;
      Cursor tc = locate(f0 + par, pre, B, Hkv);
      const float sl2 = p.scale_log2;
      for (int kk = par; kk < ntiles; kk += 2) {
        int slot;
        uint32_t parity;
        ring_pos<RING>(kk, slot, parity);
        const bool okw = mbar_wait(&full[slot], parity, p.status, p.wait_ns);
        if (!__all_sync(0xffffffffu, okw)) return;
        uint8_t* st = smem + slot * L::kStageBytes;
        const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + L::kOffKsz);
        const uint32_t* vsz = reinterpret_cast<const uint32_t*>(st + L::kOffVsz);
        const int len = lens[tc.b];
        // Lane l takes tokens 2l and 2l+1 (all G groups of each: the raw words
        // are [token][group]) and writes their entries in the consumers'
        // fragment order: warp l/8; K table rows 2(l%4) and 2(l%4)+1, slot
        // (l/4)%2 of the float4; V tables column l%4, slot (l/4)%2.  The K
        // scale carries the softmax scale (log2 domain).  The K table
        // overwrites the raw words, so all of them are read first.
        const int t0 = 2 * lane;
        const int kslot = ((lane >> 3) * 8 + 2 * (lane & 3)) * 2 + ((lane >> 2) & 1);   // float2 index in group 0
        const int vslot = ((lane >> 3) * 4 + (lane & 3)) * 2 + ((lane >> 2) & 1);       // u32 index in group 0
        uint32_t kw[2][G], vw[2][G];
        load_words<G>(kw[0], ksz + t0 * G);
        load_words<G>(kw[1], ksz + (t0 + 1) * G);
        load_words<G>(vw[0], vsz + t0 * G);
        load_words<G>(vw[1], vsz + (t0 + 1) * G);
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (tc.i * kTile + t0 + u >= len) {   // past the sequence end: zero scales
#pragma unroll
            for (int grp = 0; grp < G; ++grp) kw[u][grp] = vw[u][grp] = 0u;
          }
        __syncwarp();
        float2* ktab = reinterpret_cast<float2*>(st + L::kOffKt);
        uint32_t* vts = reinterpret_cast<uint32_t*>(st + L::kOffVtS);
        uint32_t* vtz = reinterpret_cast<uint32_t*>(st + L::kOffVtZ);
#pragma unroll
        for (int grp = 0; grp < G; ++grp) {
          const float ks0 = half_lo(kw[0][grp]) * sl2, ks1 = half_lo(kw[1][grp]) * sl2;
          ktab[grp * kTile + kslot] = make_float2(ks0, (1024.0f + half_hi(kw[0][grp])) * ks0);
          ktab[grp * kTile + kslot + 2] = make_float2(ks1, (1024.0f + half_hi(kw[1][grp])) * ks1);
          vts[grp * (kTile / 2) + vslot] = scale_pair(vw[0][grp], vw[1][grp]);
          vtz[grp * (kTile / 2) + vslot] = zero_biased_pair(vw[0][grp], vw[1][grp]);
        }
        // the raw-word area is refilled by TMA (async proxy) once the stage is released
        fence_proxy_async_smem();
        if (lane == 0) {
          const int n_b = pre[tc.b + 1] - pre[tc.b];
          int flags = tc.i;
          if (p.bits[tc.kvh] == 4) flags |= kFlag4;
          if ((tc.i + 1) * kTile <= len) flags |= kFlagFull;
          if (tc.i == 0 || kk == 0) flags |= kFlagStart;
          if (tc.i == n_b - 1 || kk == ntiles - 1) flags |= kFlagEnd;
          *reinterpret_cast<int4*>(st + L::kOffMeta) = make_int4(tc.b, tc.kvh, flags, len);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[slot]);
        advance(tc, pre, B, Hkv);
        if (kk + 2 < ntiles) advance(tc, pre, B, Hkv);
      }
      return;
    }
    if (w == kWarps + 2) {
      // ---------------- epilogue warp: every piece end but the CTA's last ----------------
      zero_empty_rows<D>(p, lens, lane);
      const int npieces = count_pieces(f0, ntiles, pre, B, Hkv);
      for (int e = 0; e + 1 < npieces; ++e) {
        const bool okw = mbar_wait(epi_full, e & 1, p.status, p.wait_ns);
        if (!__all_sync(0xffffffffu, okw)) return;
        const int4 info = eb->info;
        segment_end<D, 8>(p, eb, &eb->flag[0], info.x, info.y, pre, N, C, lane, 32, WarpSync{}, epi_empty);
      }
      return;
    }
    return;
  }

  // ---------------- consumers: four warps ----------------
  tc::reg_alloc<kConsumerRegs>();
  const LaneAddr la = lane_addr<D>(w, lane);
  uint32_t qa[D / 16][2];
  float qs[G][2];   // per-group sums of q for heads 2t, 2t+1
  float O[D / 16][4];
  float Z[2][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  bool ok = true;
  int n_end = 0;
  uint32_t gphase = 0;

  for (int k = 0; k < ntiles;) {
    int slot, slot1 = 0;
    uint32_t parity;
    ring_pos<RING>(k, slot, parity);
    ok = ok && mbar_wait(&ready[slot], parity, p.status, p.wait_ns);
    if (!ok) break;   // a timed-out wait ends this warp (status already set)
    const uint8_t* st0 = smem + slot * L::kStageBytes;
    const int4 meta = *reinterpret_cast<const int4*>(st0 + L::kOffMeta);
    const int cb = meta.x, ckvh = meta.y, len = meta.w;
    const bool four = (meta.z & kFlag4) != 0;
    if (meta.z & kFlagStart) {
      float qsum[G];
      load_q<D>(qa, qsum, p, reinterpret_cast<const uint16_t*>(st0 + L::kOffQ), four ? 4 : 8, g, t);
#pragma unroll
      for (int grp = 0; grp < G; ++grp) {
        qs[grp][0] = __shfl_sync(0xffffffffu, qsum[grp], (2 * t) << 2);
        qs[grp][1] = __shfl_sync(0xffffffffu, qsum[grp], (2 * t + 1) << 2);
      }
#pragma unroll
      for (int i = 0; i < D / 16; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.0f;
#pragma unroll
      for (int z = 0; z < 2; ++z) Z[z][0] = Z[z][1] = Z[z][2] = Z[z][3] = 0.0f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.0f;
    }
    // tokens of a tile inside the sequence
    auto tile_lim = [len](int f) { return (f & kFlagFull) ? kTile : len - (f & 0xFFFFFF) * kTile; };
    int fend, nt;
    if (!(meta.z & kFlagEnd)) {
      // the next tile belongs to the same piece: take both in one step
      uint32_t parity1;
      ring_pos<RING>(k + 1, slot1, parity1);
      ok = ok && mbar_wait(&ready[slot1], parity1, p.status, p.wait_ns);
      if (!ok) break;
      const uint8_t* st1 = smem + slot1 * L::kStageBytes;
      const int f1 = reinterpret_cast<const int4*>(st1 + L::kOffMeta)->z;
      const uint32_t ss[2] = {smem_u32(st0), smem_u32(st1)};
      const uint8_t* const sp[2] = {st0, st1};
      const int lim[2] = {tile_lim(meta.z), tile_lim(f1)};
      if (!four) consume_tiles<D, 8, 2>(ss, sp, lim, qa, qs, O, Z, m_run, l_run, la, w, g, t);
      else consume_tiles<D, 4, 2>(ss, sp, lim, qa, qs, O, Z, m_run, l_run, la, w, g, t);
      fend = f1;
      nt = 2;
    } else {
      const uint32_t ss[1] = {smem_u32(st0)};
      const uint8_t* const sp[1] = {st0};
      const int lim[1] = {tile_lim(meta.z)};
      if (!four) consume_tiles<D, 8, 1>(ss, sp, lim, qa, qs, O, Z, m_run, l_run, la, w, g, t);
      else consume_tiles<D, 4, 1>(ss, sp, lim, qa, qs, O, Z, m_run, l_run, la, w, g, t);
      fend = meta.z;
      nt = 1;
    }

    // ---- end of a piece: the warps' states go to the hand-off buffer ----
    if (fend & kFlagEnd) {
      // sums over the warp's tokens (rows g) for heads 2t, 2t+1
      float l_tot[2] = {l_run[0], l_run[1]};
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l_tot[0] += __shfl_xor_sync(0xffffffffu, l_tot[0], o);
        l_tot[1] += __shfl_xor_sync(0xffffffffu, l_tot[1], o);
      }
      if (n_end > 0) ok = ok && mbar_wait(epi_empty, (n_end - 1) & 1, p.status, p.wait_ns);
      if (!ok) break;
      if (g == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (2 * t + e < p.rep) {
            eb->ml[w][2 * t + e][0] = m_run[e];
            eb->ml[w][2 * t + e][1] = l_tot[e];
          }
      }
#pragma unroll
      for (int grp = 0; grp < G; ++grp) {
        // zero-point term of group grp for heads 2t, 2t+1 sits in row grp of Z[grp & 1]
        const float r0 = __shfl_sync(0xffffffffu, Z[grp & 1][0], grp * 4 + t);
        const float r1 = __shfl_sync(0xffffffffu, Z[grp & 1][1], grp * 4 + t);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * t + e;
          const float r = e ? r1 : r0;
          if (h < p.rep) {
            float* dst = eb->o[w][h];
#pragma unroll
            for (int mh = 0; mh < 2; ++mh)
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const int ch = four ? acc_channel<4>(grp, mh, half, g) : acc_channel<8>(grp, mh, half, g);
                dst[ch] = O[2 * grp + mh][2 * half + e] - r;
              }
          }
        }
      }
      ++n_end;
      if (k + nt < ntiles) {
        // not the CTA's last piece: the epilogue warp takes it from here
        if (w == 0 && lane == 0) eb->info = make_int4(cb, ckvh, 0, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_full);
      } else {
        // the last piece: the CTA has no more tiles, so the four consumer
        // warps finish it themselves
        const ConsumerSync cs{gbar, &gphase, &ok, p.status, p.wait_ns};
        cs();
        segment_end<D, 8>(p, eb, &eb->flag[1], cb, ckvh, pre, N, C, tid, kWarps * 32, cs, nullptr);
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[slot]);
      if (nt == 2) mbar_arrive(&empty[slot1]);
    }
    k += nt;
  }
}

// CTAs per SM of the decode kernel on the current device (the same for both
// ring depths: their resources are the same); sets the shared-memory limit
// of both instantiations once per device.
template <int D, bool PAGED>
int ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    const size_t sm = Smem<D>::bytes(64);
    const int lim = static_cast<int>(Smem<D>::bytes(4096));
    cudaFuncSetAttribute(decode_split_kernel<D, PAGED, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    cudaFuncSetAttribute(decode_split_kernel<D, PAGED, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<D, PAGED, kStages>, kThreads, sm) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// The register split inside the kernel assumes 128 registers per thread at
// launch; any other count would make the consumers' setmaxnreg wait forever.
template <int D, bool PAGED>
bool regs_ok() {
  static int cached = -1;
  if (cached < 0) {
    cudaFuncAttributes fa, fb;
    cached = (cudaFuncGetAttributes(&fa, decode_split_kernel<D, PAGED, 2>) == cudaSuccess && fa.numRegs == 128 &&
              cudaFuncGetAttributes(&fb, decode_split_kernel<D, PAGED, kStages>) == cudaSuccess && fb.numRegs == 128)
                 ? 1
                 : 0;
  }
  return cached == 1;
}

// Launched with programmatic stream serialization: the kernel's CTAs may be
// scheduled while the previous kernel of the stream drains; the kernel waits
// for it (griddepcontrol.wait) before its first global memory access.
template <int D, bool PAGED>
cudaError_t launch_split(const DParams& p, int C, int B, int ring, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D>::bytes(B);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return ring == 2 ? cudaLaunchKernelEx(&cfg, decode_split_kernel<D, PAGED, 2>, p)
                   : cudaLaunchKernelEx(&cfg, decode_split_kernel<D, PAGED, kStages>, p);
}

}  // namespace

int decode_num_ctas(int D) {
  // the paged instantiations have the same resources (checked by regs_ok)
  const int per = D == 128 ? ctas_per_sm<128, false>() : ctas_per_sm<64, false>();
  return device_sm_count() * per;
}

// workspace: [cnt: B*Hkv int32, padded to 16 B][lse: slots*rep f32, padded][o: slots*rep*D f32]
static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

size_t decode_workspace_counter_bytes(int B, int Hkv) { return align16(static_cast<size_t>(B) * Hkv * 4); }

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int D, int num_ctas) {
  const size_t rep = static_cast<size_t>(Hq / Hkv);
  const size_t slots = static_cast<size_t>(B) * Hkv + num_ctas;
  return align16(static_cast<size_t>(B) * Hkv * 4) + align16(slots * rep * 4) + slots * rep * D * 4;
}

kvq_status launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const kvq_cache& K = *a.k;
  const kvq_cache& Vc = *a.v;
  // K.B x K.Tcap is the storage (a page pool when a block table is given);
  // B x Tcap the sequences and their capacity
  const int D = K.D, Hkv = K.Hkv;
  const int B = a.bt != nullptr ? a.bt_B : K.B;
  const int Tcap = a.bt != nullptr ? a.bt_max_pages * kTile : K.Tcap;
  if (B > 4096) return KVQ_ERR_UNSUPPORTED;  // dynamic shared memory was sized for B <= 4096
  const bool paged = a.bt != nullptr;
  const bool regs = D == 128 ? (paged ? regs_ok<128, true>() : regs_ok<128, false>())
                             : (paged ? regs_ok<64, true>() : regs_ok<64, false>());
  if (!regs) return KVQ_ERR_UNSUPPORTED;
  const int C = decode_num_ctas(D);
  const size_t need = decode_workspace_bytes(B, a.Hq, Hkv, D, C);
  if (a.ws == nullptr || a.ws_bytes < need) return KVQ_ERR_WORKSPACE;

  DParams p;
  memset(&p, 0, sizeof(p));
  const HeadLayout& hl = a.layout;
  const uint64_t rows8 = static_cast<uint64_t>(hl.n8) * K.B * K.Tcap;
  const uint64_t rows4 = static_cast<uint64_t>(hl.n4) * K.B * K.Tcap;
  auto enc = [&](CUtensorMap* m, const uint8_t* base, int bits, uint64_t rows) -> bool {
    if (rows == 0) return true;
    const uint32_t R = static_cast<uint32_t>(D * bits / 8);
    const CUtensorMapSwizzle sw = R == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : R == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
    return encode_tensor_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, R, rows, R, R, kTile, sw) ==
           CUDA_SUCCESS;
  };
  if (!enc(&p.tm_k8, K.codes, 8, rows8) || !enc(&p.tm_k4, K.codes + hl.off4, 4, rows4) ||
      !enc(&p.tm_v8, Vc.codes, 8, rows8) || !enc(&p.tm_v4, Vc.codes + hl.off4, 4, rows4))
    return KVQ_ERR_CUDA;
  p.k_sz = K.sz;
  p.v_sz = Vc.sz;
  p.q = a.q;
  p.seq_lens = a.seq_lens;
  const int rep = a.Hq / Hkv;
  const size_t slots = static_cast<size_t>(B) * Hkv + C;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const size_t cnt_bytes = align16(static_cast<size_t>(B) * Hkv * 4);
  p.ws_cnt = reinterpret_cast<int32_t*>(ws);
  p.ws_lse = reinterpret_cast<float*>(ws + cnt_bytes);
  p.ws_o = reinterpret_cast<float*>(ws + cnt_bytes + align16(slots * rep * 4));
  p.out = a.out;
  p.status = a.status;
  p.out_dtype = a.out_dtype;
  p.B = B; p.Hq = a.Hq; p.Hkv = Hkv; p.Tcap = Tcap; p.rep = rep; p.num_ctas = C;
  p.bt = a.bt;
  p.bt_stride = a.bt_max_pages;
  p.pB = K.B;
  p.pT = K.Tcap;
  const float scale = a.softmax_scale > 0.0f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane[h] = hl.plane_idx[h];
    p.bits[h] = hl.bits[h];
  }
  const int ring = a.pol.ring;
  p.l2_warm = a.pol.l2_warm;
  p.issue_limit = a.pol.issue_limit;
  p.wait_ns = a.pol.wait_ns;
  if ((ring != 2 && ring != kStages) || p.l2_warm < 0 || p.l2_warm > kMaxL2Tiles || p.wait_ns == 0)
    return KVQ_ERR_INVALID_ARG;
  if (paged) (void)(D == 128 ? ctas_per_sm<128, true>() : ctas_per_sm<64, true>());   // sets its smem limit
  const cudaError_t e =
      D == 128 ? (paged ? launch_split<128, true>(p, C, B, ring, stream) : launch_split<128, false>(p, C, B, ring, stream))
               : (paged ? launch_split<64, true>(p, C, B, ring, stream) : launch_split<64, false>(p, C, B, ring, stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
