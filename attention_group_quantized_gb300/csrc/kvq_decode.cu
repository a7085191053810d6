// kvq_decode.cu -- decode attention over the group-quantised KV cache.
//
// Method: one query token per (sequence, query head) attends its sequence's
// cached keys; the cache holds integer codes with a per-group fp16 scale and
// zero point (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.4), and
// dequantisation happens inside the attention read (same page, §1.3).  The
// keys are visited tile by tile with an online softmax carrying the running
// max and normaliser (same page, §2.2); splits of the key range run on
// different CTAs and a second pass merges them by log-sum-exp.
//
// GB300 design (HBM-bound):
//  * Stream-K split: the (sequence, KV head, 64-token tile) work list is cut
//    into equal contiguous ranges, one per persistent CTA (SMs x CTAs/SM), so
//    ragged lengths cost no load imbalance; each CTA emits one partial
//    (o, lse) per segment piece it touched.
//  * A producer warp streams each tile's codes by TMA (2D tensor copies with
//    hardware swizzle, so the fragment reads below are bank-conflict free)
//    and its scale/zero words by 1D bulk copies into a 3-stage ring; per-slot
//    full/empty mbarriers let the four consumer warps run independently.
//  * The products run on the tensor cores with exact integer operands: a code
//    byte becomes the fp16 value 1024 + c by a byte permute, and one fp16
//    subtraction of (1024 + z) gives c - z exactly.
//      S = Q K^T: rows = the query heads of the KV head, columns = tokens;
//        Q.(c - z) is summed per group of 32 channels and scaled by the
//        group's fp32 scale.
//      O^T = V^T P^T: rows = channels, columns = query heads; the channel's
//        scale is applied in fp16 ((c - z) * s, one rounding), and P comes
//        straight from the S accumulator registers (same fragment layout).
//  * One CTA serves all query heads of a KV head, so every cache byte is read
//    once for the whole GQA group.
#include <cfloat>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTile = 64;       // tokens per pipeline stage
constexpr int kWarps = 4;       // consumer warps; each owns 16 tokens of a tile
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kMaxRep = 8;      // query heads per KV head

struct DParams {
  CUtensorMap tm_k8, tm_k4, tm_v8, tm_v4;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  const uint16_t* q;
  const int32_t* seq_lens;
  int32_t* ws_pre;      // [B+1] tile prefix sums, written by CTA 0 for the merge
  float* ws_lse;        // [slots][rep]
  float* ws_o;          // [slots][rep][D]
  void* out;
  int32_t* status;
  int32_t out_dtype;
  int32_t B, Hq, Hkv, Tcap, rep, num_ctas;
  float scale_log2;
  int32_t plane[KVQ_MAX_HKV];
  int8_t bits[KVQ_MAX_HKV];
};

template <int D>
struct Smem {
  static constexpr int G = D / 32;
  static constexpr int kCodeBytes = kTile * D;          // room for an 8-bit tile
  static constexpr int kSzBytes = kTile * G * 4;
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kSzBytes;
  // a finished slot doubles as the merge scratch of a piece end
  static constexpr int kMergeO = kWarps * kMaxRep * D * 4;
  static_assert(kMergeO + kWarps * kMaxRep * 8 <= kStageBytes, "merge scratch must fit a stage");
  static constexpr int kBars = (2 * kStages + 1) * 8;
  static constexpr int kFixed = kStages * kStageBytes + kBars;
  static size_t bytes(int B) { return 1024 + kFixed + static_cast<size_t>(B + 1) * 4 * 2; }
};

// Byte offset of (row, byte) inside a TMA tile written with the swizzle mode
// matching its row pitch R (128B, 64B or 32B): the 16-byte chunk index is
// XORed with address bits 7.. of the row start.
template <int R>
__device__ __forceinline__ uint32_t swz(int row, int byte) {
  if constexpr (R == 128) return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
  if constexpr (R == 64) return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15));
  return row * 32 + ((((byte >> 4) ^ ((row >> 2) & 1)) << 4) | (byte & 15));
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(base + off);
}
__device__ __forceinline__ uint2 lds64(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const uint2*>(base + off);
}
__device__ __forceinline__ uint4 lds128(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const uint4*>(base + off);
}

// Position in the flat work list: sequence b, KV head, tile index i.
struct Cursor {
  int b, kvh, i;
};

__device__ __forceinline__ void advance(Cursor& c, const int32_t* pre, int B, int Hkv) {
  const int n = pre[c.b + 1] - pre[c.b];
  if (++c.i < n) return;
  c.i = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < B && pre[c.b + 1] == pre[c.b]);
}

__device__ __forceinline__ Cursor locate(int64_t f, const int32_t* pre, int B, int Hkv) {
  // largest b with Hkv * pre[b] <= f; it is a non-empty sequence because f < Hkv * pre[B]
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(Hkv) * pre[mid] <= f) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int n = pre[b + 1] - pre[b];
  const int64_t off = f - static_cast<int64_t>(Hkv) * pre[b];
  Cursor c;
  c.b = b;
  c.kvh = static_cast<int>(off / n);
  c.i = static_cast<int>(off % n);
  return c;
}

// Q fragments for S = Q K^T (A operand rows = query heads of the group, zero
// from rep up), channel order matching the code unpacking of the bit-width.
template <int D>
__device__ __forceinline__ void load_q(uint32_t (&qa)[D / 32][2][2], const DParams& p, int b, int kvh,
                                       int bits, int g, int t) {
  constexpr int G = D / 32;
#pragma unroll
  for (int grp = 0; grp < G; ++grp) {
    float f[8];
    if (g < p.rep) {
      const uint16_t* src = p.q + (static_cast<int64_t>(b) * p.Hq + kvh * p.rep + g) * D + grp * 32 + t * 8;
      const uint4 raw = *reinterpret_cast<const uint4*>(src);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      bool ok = true;
#pragma unroll
      for (int i = 0; i < 8; ++i) ok &= fabsf(f[i]) < 65504.0f;
      if (!ok) report(p.status, KVQ_ERR_NONFINITE);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.0f;
    }
    if (bits == 8) {  // byte order: k-step 0 = ch 0..3, k-step 1 = ch 4..7
      qa[grp][0][0] = pack_half2(f[0], f[1]);
      qa[grp][0][1] = pack_half2(f[2], f[3]);
      qa[grp][1][0] = pack_half2(f[4], f[5]);
      qa[grp][1][1] = pack_half2(f[6], f[7]);
    } else {          // nibble order: (0,4)(1,5) then (2,6)(3,7)
      qa[grp][0][0] = pack_half2(f[0], f[4]);
      qa[grp][0][1] = pack_half2(f[1], f[5]);
      qa[grp][1][0] = pack_half2(f[2], f[6]);
      qa[grp][1][1] = pack_half2(f[3], f[7]);
    }
  }
}

// Scores of one warp's 16 tokens for head row g: S[j][e] belongs to token
// 16w + 8j + 2t + e of the tile.  Thread (g, t) feeds the codes of token
// 16w + 8j + g (B operand) and receives the scores of tokens 8j + 2t + e.
template <int D, int BITS>
__device__ __forceinline__ void qk_tile(float (&S)[2][2], const uint32_t (&qa)[D / 32][2][2],
                                        const uint8_t* kc, const uint32_t* ksz, int w, int g, int t) {
  constexpr int G = D / 32;
  constexpr int R = D * BITS / 8;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = 16 * w + 8 * j + g;
    const int ta = 16 * w + 8 * j + 2 * t;
    uint32_t zrow[G], s0[G], s1[G];
    if constexpr (G == 4) {
      const uint4 a = *reinterpret_cast<const uint4*>(ksz + row * 4);
      const uint4 b0 = *reinterpret_cast<const uint4*>(ksz + ta * 4);
      const uint4 b1 = *reinterpret_cast<const uint4*>(ksz + (ta + 1) * 4);
      zrow[0] = a.x; zrow[1] = a.y; zrow[2] = a.z; zrow[3] = a.w;
      s0[0] = b0.x; s0[1] = b0.y; s0[2] = b0.z; s0[3] = b0.w;
      s1[0] = b1.x; s1[1] = b1.y; s1[2] = b1.z; s1[3] = b1.w;
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(ksz + row * 2);
      const uint2 b0 = *reinterpret_cast<const uint2*>(ksz + ta * 2);
      const uint2 b1 = *reinterpret_cast<const uint2*>(ksz + (ta + 1) * 2);
      zrow[0] = a.x; zrow[1] = a.y;
      s0[0] = b0.x; s0[1] = b0.y;
      s1[0] = b1.x; s1[1] = b1.y;
    }
    float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      const uint32_t zb = zero_biased2(zrow[grp]);
      float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (BITS == 8) {
        const uint2 cw = lds64(kc, swz<R>(row, grp * 32 + t * 8));
        mma_16816(c, qa[grp][0][0], 0u, qa[grp][0][1], 0u, hsub2_u32(bytes01_biased(cw.x), zb),
                  hsub2_u32(bytes23_biased(cw.x), zb));
        mma_16816(c, qa[grp][1][0], 0u, qa[grp][1][1], 0u, hsub2_u32(bytes01_biased(cw.y), zb),
                  hsub2_u32(bytes23_biased(cw.y), zb));
      } else {
        const uint32_t cw = lds32(kc, swz<R>(row, grp * 16 + t * 4));
        mma_16816(c, qa[grp][0][0], 0u, qa[grp][0][1], 0u, hsub2_u32(nib_biased(cw), zb),
                  hsub2_u32(nib_biased(cw >> 4), zb));
        mma_16816(c, qa[grp][1][0], 0u, qa[grp][1][1], 0u, hsub2_u32(nib_biased(cw >> 8), zb),
                  hsub2_u32(nib_biased(cw >> 12), zb));
      }
      acc0 = fmaf(half_lo(s0[grp]), c[0], acc0);
      acc1 = fmaf(half_lo(s1[grp]), c[1], acc1);
    }
    S[j][0] = acc0;
    S[j][1] = acc1;
  }
}

// O^T[ch][h] += V_hat^T[ch][tok] P^T[tok][h] over the warp's 16 tokens.
// A operand (rows = channels, k = tokens): thread (g, t) supplies channels
// CPT*g + m (row g of m-tile m) and CPT*g + CPT/2 + m (row g + 8), CPT = D/8,
// of tokens 2t, 2t+1 (k 0..7) and 8+2t, 9+2t (k 8..15).  B operand (k =
// tokens, n = heads) is P straight from the score fragments.  Accumulator
// O[m]: c0/c1 = heads 2t, 2t+1 of the row-g channel, c2/c3 of the row-(g+8)
// channel.  Tokens past the sequence end read as s = 0, z = 0, so stale
// cache words cannot poison O.
template <int D, int BITS>
__device__ __forceinline__ void pv_tile(float (&O)[D / 16][4], const uint32_t (&pb)[2], const uint8_t* vc,
                                        const uint32_t* vsz, const bool (&valid)[2][2], int w, int g, int t) {
  constexpr int G = D / 32;
  constexpr int R = D * BITS / 8;
  constexpr int CPT = D / 8;            // channels per thread (16 or 8)
  constexpr int HALF = CPT / 2;         // channels per row half = m-tiles
  const int grp = (g * CPT) / 32;       // all of a thread's channels share one group
  int rows[2][2];
  uint32_t word[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      rows[j][e] = 16 * w + 8 * j + 2 * t + e;
      word[j][e] = valid[j][e] ? vsz[rows[j][e] * G + grp] : 0u;
    }
  // (s_a, s_b) and (1024 + z_a, 1024 + z_b) for the token pairs j = 0, 1
  uint32_t s2[2], zb[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    s2[j] = prmt(word[j][0], word[j][1], 0x5410u);
    zb[j] = zero_biased_pair(word[j][0], word[j][1]);
  }
  // exact (c - z) then one fp16 rounding of (c - z) * s, for a token pair
  auto deq = [&](uint32_t biased, int j) -> uint32_t {
    uint32_t d = hsub2_u32(biased, zb[j]);
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&d), *reinterpret_cast<const __half2*>(&s2[j]));
    return *reinterpret_cast<uint32_t*>(&r);
  };
  uint32_t A[2][2][HALF];   // [token pair j][row half][m]
  if constexpr (BITS == 8) {
    // per token: CPT bytes = channels [CPT*g, CPT*g + CPT), word wi = channels 4wi .. 4wi+3
    uint32_t wv[2][2][CPT / 4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if constexpr (CPT == 16) {
          const uint4 v = lds128(vc, swz<R>(rows[j][e], g * 16));
          wv[j][e][0] = v.x; wv[j][e][1] = v.y; wv[j][e][2] = v.z; wv[j][e][3] = v.w;
        } else {
          const uint2 v = lds64(vc, swz<R>(rows[j][e], g * 8));
          wv[j][e][0] = v.x; wv[j][e][1] = v.y;
        }
      }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int wq = 0; wq < HALF / 4; ++wq) {
          const int wi = hr * (HALF / 4) + wq;
          const uint32_t x0 = prmt(wv[j][0][wi], wv[j][1][wi], 0x5140u);  // bytes 0,1 of both tokens
          const uint32_t x1 = prmt(wv[j][0][wi], wv[j][1][wi], 0x7362u);  // bytes 2,3
          A[j][hr][4 * wq + 0] = deq(bytes01_biased(x0), j);
          A[j][hr][4 * wq + 1] = deq(bytes23_biased(x0), j);
          A[j][hr][4 * wq + 2] = deq(bytes01_biased(x1), j);
          A[j][hr][4 * wq + 3] = deq(bytes23_biased(x1), j);
        }
  } else {
    // per token: CPT/2 bytes; nibble n of the thread's chunk = channel CPT*g + n
    uint32_t wv[2][2][CPT / 8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if constexpr (CPT == 16) {
          const uint2 v = lds64(vc, swz<R>(rows[j][e], g * 8));
          wv[j][e][0] = v.x; wv[j][e][1] = v.y;
        } else {
          wv[j][e][0] = lds32(vc, swz<R>(rows[j][e], g * 4));
        }
      }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int base = hr * HALF;                  // first nibble of this row half
        const int sh = (base % 8) * 4;
        const uint32_t a0 = wv[j][0][base / 8] >> sh, a1 = wv[j][1][base / 8] >> sh;
        const uint32_t ev0 = a0 & 0x0F0F0F0Fu, ev1 = a1 & 0x0F0F0F0Fu;                // nibbles 0,2,4,6
        const uint32_t od0 = (a0 >> 4) & 0x0F0F0F0Fu, od1 = (a1 >> 4) & 0x0F0F0F0Fu;  // nibbles 1,3,5,7
        const uint32_t e01 = prmt(ev0, ev1, 0x5140u), o01 = prmt(od0, od1, 0x5140u);
        A[j][hr][0] = deq(bytes01_biased(e01), j);
        A[j][hr][1] = deq(bytes01_biased(o01), j);
        A[j][hr][2] = deq(bytes23_biased(e01), j);
        A[j][hr][3] = deq(bytes23_biased(o01), j);
        if constexpr (HALF == 8) {
          const uint32_t e23 = prmt(ev0, ev1, 0x7362u), o23 = prmt(od0, od1, 0x7362u);
          A[j][hr][4] = deq(bytes01_biased(e23), j);
          A[j][hr][5] = deq(bytes01_biased(o23), j);
          A[j][hr][6] = deq(bytes23_biased(e23), j);
          A[j][hr][7] = deq(bytes23_biased(o23), j);
        }
      }
  }
#pragma unroll
  for (int m = 0; m < HALF; ++m) mma_16816(O[m], A[0][0][m], A[0][1][m], A[1][0][m], A[1][1][m], pb[0], pb[1]);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3) decode_split_kernel(const __grid_constant__ DParams p) {
  using L = Smem<D>;
  constexpr int G = D / 32;
  constexpr int CPT = D / 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * L::kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* gbar = empty + kStages;       // consumer-group barrier for piece ends
  int32_t* pre = reinterpret_cast<int32_t*>(smem + L::kFixed);
  int32_t* lens = pre + (p.B + 1);

  // let the merge grid get scheduled early; it waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;");

  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int B = p.B, Hkv = p.Hkv;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(gbar, kWarps);
    fence_barrier_init();
  }
  for (int b = tid; b < B; b += blockDim.x) {
    int L0 = p.seq_lens[b];
    if (L0 < 0 || L0 > p.Tcap) {
      report(p.status, KVQ_ERR_INVALID_ARG);
      L0 = L0 < 0 ? 0 : p.Tcap;
    }
    lens[b] = L0;
  }
  __syncthreads();
  if (w == 0) {  // per-sequence tile counts and their prefix sums
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = b < B ? (lens[b] + kTile - 1) / kTile : 0;
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
  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += blockDim.x) p.ws_pre[b] = pre[b];

  const int64_t N = static_cast<int64_t>(Hkv) * pre[B];
  const int C = p.num_ctas;
  const int64_t f0 = N * blockIdx.x / C;
  const int64_t f1 = N * (blockIdx.x + 1) / C;
  const int ntiles = static_cast<int>(f1 - f0);
  if (ntiles <= 0) return;

  if (w == kWarps) {
    // ---------------- producer warp: one thread streams the tiles ----------------
    if (lane != 0) return;
    Cursor pc = locate(f0, pre, B, Hkv);
    for (int k = 0; k < ntiles; ++k) {
      const int slot = k % kStages;
      if (k >= kStages && !mbar_wait(&empty[slot], ((k / kStages) - 1) & 1, p.status)) return;
      uint8_t* st = smem + slot * L::kStageBytes;
      const int bits = p.bits[pc.kvh];
      const int R = D * bits / 8;
      const int32_t row0 = (p.plane[pc.kvh] * B + pc.b) * p.Tcap + pc.i * kTile;
      const int64_t szoff = (static_cast<int64_t>(pc.kvh) * B + pc.b) * p.Tcap + static_cast<int64_t>(pc.i) * kTile;
      uint64_t* bar = &full[slot];
      mbar_arrive_expect_tx(bar, 2 * kTile * R + 2 * L::kSzBytes);
      tma_2d_g2s(st, bits == 8 ? &p.tm_k8 : &p.tm_k4, 0, row0, bar);
      tma_2d_g2s(st + L::kCodeBytes, bits == 8 ? &p.tm_v8 : &p.tm_v4, 0, row0, bar);
      bulk_g2s(st + 2 * L::kCodeBytes, p.k_sz + szoff * G, L::kSzBytes, bar);
      bulk_g2s(st + 2 * L::kCodeBytes + L::kSzBytes, p.v_sz + szoff * G, L::kSzBytes, bar);
      advance(pc, pre, B, Hkv);
    }
    return;
  }

  // ---------------- consumers: four warps ----------------
  Cursor cc = locate(f0, pre, B, Hkv);
  uint32_t qa[G][2][2];
  float O[D / 16][4];
  float m_run = -INFINITY, l_run = 0.0f;
  bool piece_start = true;
  bool ok = true;
  uint32_t gphase = 0;
  // bounded barrier among the four consumer warps (a plain bar.sync could wait forever
  // if one warp left after a timed-out wait)
  auto group_sync = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(gbar);
    ok = ok && mbar_wait(gbar, gphase & 1, p.status);
    ++gphase;
    __syncwarp();
  };

  for (int k = 0; k < ntiles; ++k) {
    const int slot = k % kStages;
    const int bits = p.bits[cc.kvh];
    const int n_b = pre[cc.b + 1] - pre[cc.b];
    if (piece_start) {
      load_q<D>(qa, p, cc.b, cc.kvh, bits, g, t);
#pragma unroll
      for (int i = 0; i < D / 16; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.0f;
      m_run = -INFINITY;
      l_run = 0.0f;
    }
    ok = ok && mbar_wait(&full[slot], (k / kStages) & 1, p.status);
    if (!ok) break;   // a timed-out wait ends this warp (status already set)
    uint8_t* st = smem + slot * L::kStageBytes;
    const uint8_t* kc = st;
    const uint8_t* vc = st + L::kCodeBytes;
    const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + 2 * L::kCodeBytes);
    const uint32_t* vsz = reinterpret_cast<const uint32_t*>(st + 2 * L::kCodeBytes + L::kSzBytes);

    float S[2][2];
    if (bits == 8) qk_tile<D, 8>(S, qa, kc, ksz, w, g, t);
    else qk_tile<D, 4>(S, qa, kc, ksz, w, g, t);

    // mask past the sequence end, move to the log2 domain, online softmax per head row g
    const int len = lens[cc.b];
    bool valid[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        valid[j][e] = cc.i * kTile + 16 * w + 8 * j + 2 * t + e < len;
        S[j][e] = valid[j][e] ? S[j][e] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, S[j][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.0f : m_new;
    const float alpha = fast_exp2(m_run - m_use);
    float P[2][2];
    float psum = 0.0f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        P[j][e] = fast_exp2(S[j][e] - m_use);
        psum += P[j][e];
      }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (__any_sync(0xffffffffu, alpha != 1.0f)) {
      // O^T columns are heads 2t, 2t+1; their factors live in rows g = 2t, 2t+1
      const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * t) << 2);
      const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) << 2);
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        O[i][0] *= a0; O[i][1] *= a1;
        O[i][2] *= a0; O[i][3] *= a1;
      }
    }
    const uint32_t pb[2] = {pack_half2(P[0][0], P[0][1]), pack_half2(P[1][0], P[1][1])};
    if (bits == 8) pv_tile<D, 8>(O, pb, vc, vsz, valid, w, g, t);
    else pv_tile<D, 4>(O, pb, vc, vsz, valid, w, g, t);

    // ---- end of a piece: merge the four warps and write the partial ----
    const bool piece_end = (cc.i == n_b - 1) || (k == ntiles - 1);
    if (piece_end) {
      float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
      float* m_o = reinterpret_cast<float*>(st);                 // this slot, once every warp is done with it
      float* m_ml = reinterpret_cast<float*>(st + L::kMergeO);
      group_sync();
      if (t == 0 && g < p.rep) {
        m_ml[(w * kMaxRep + g) * 2 + 0] = m_run;
        m_ml[(w * kMaxRep + g) * 2 + 1] = l_tot;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * t + e;
        if (h < p.rep) {
          float* dst = m_o + (w * kMaxRep + h) * D;
#pragma unroll
          for (int m = 0; m < D / 16; ++m) {
            dst[CPT * g + m] = O[m][e];
            dst[CPT * g + CPT / 2 + m] = O[m][2 + e];
          }
        }
      }
      group_sync();
      const int slotw = cc.b * Hkv + cc.kvh + blockIdx.x;
      for (int idx = tid; idx < p.rep * D; idx += kWarps * 32) {
        const int h = idx / D, ch = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, m_ml[(ww * kMaxRep + h) * 2]);
        float Lsum = 0.0f, o = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int ww = 0; ww < kWarps; ++ww) {
            const float sc = fast_exp2(m_ml[(ww * kMaxRep + h) * 2] - M);
            Lsum += m_ml[(ww * kMaxRep + h) * 2 + 1] * sc;
            o += m_o[(ww * kMaxRep + h) * D + ch] * sc;
          }
        }
        const bool any = M != -INFINITY && Lsum > 0.0f;
        p.ws_o[(static_cast<int64_t>(slotw) * p.rep + h) * D + ch] = any ? o / Lsum : 0.0f;
        if (ch == 0) p.ws_lse[static_cast<int64_t>(slotw) * p.rep + h] = any ? M + __log2f(Lsum) : -INFINITY;
      }
      group_sync();                                              // scratch read before the slot is refilled
      piece_start = true;
    } else {
      piece_start = false;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    advance(cc, pre, B, Hkv);
    if (!ok) break;
  }
}

// One warp per (sequence, query head): log-sum-exp merge of the partials.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const __grid_constant__ DParams p) {
  constexpr int V = D / 32;  // channels per lane
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= p.B * p.Hq) return;
  const int b = gw / p.Hq, hq = gw % p.Hq;
  const int kvh = hq / p.rep, r = hq % p.rep;
  const int B = p.B, Hkv = p.Hkv, C = p.num_ctas;
  const int32_t* pre = p.ws_pre;
  const int n_b = pre[b + 1] - pre[b];
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  if (n_b > 0) {
    const int64_t N = static_cast<int64_t>(Hkv) * pre[B];
    const int64_t start = static_cast<int64_t>(Hkv) * pre[b] + static_cast<int64_t>(kvh) * n_b;
    const int64_t last = start + n_b - 1;
    const int c0 = static_cast<int>(((start + 1) * C - 1) / N);
    const int c1 = static_cast<int>(((last + 1) * C - 1) / N);
    const int64_t seg = static_cast<int64_t>(b) * Hkv + kvh;
    // pass 1: pieces spread over the lanes -> the largest lse
    float M = -INFINITY;
    for (int c = c0 + lane; c <= c1; c += 32) {
      if (N * (c + 1) / C == N * c / C) continue;  // a CTA with an empty range wrote nothing
      M = fmaxf(M, p.ws_lse[(seg + c) * p.rep + r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // pass 2: weighted sum of the partial outputs (loads independent of each other)
    float Lsum = 0.0f;
    if (M != -INFINITY) {
      for (int c = c0; c <= c1; ++c) {
        if (N * (c + 1) / C == N * c / C) continue;
        const int64_t slot = seg + c;
        const float lse = p.ws_lse[slot * p.rep + r];
        const float wgt = lse == -INFINITY ? 0.0f : fast_exp2(lse - M);
        const float* o = p.ws_o + (slot * p.rep + r) * D + lane * V;
        if constexpr (V == 4) {
          const float4 v = *reinterpret_cast<const float4*>(o);
          acc[0] = fmaf(wgt, v.x, acc[0]); acc[1] = fmaf(wgt, v.y, acc[1]);
          acc[2] = fmaf(wgt, v.z, acc[2]); acc[3] = fmaf(wgt, v.w, acc[3]);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(o);
          acc[0] = fmaf(wgt, v.x, acc[0]); acc[1] = fmaf(wgt, v.y, acc[1]);
        }
        Lsum += wgt;
      }
      if (Lsum > 0.0f) {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] /= Lsum;
      }
    }
  }
  const int64_t orow = (static_cast<int64_t>(b) * p.Hq + hq) * D + lane * V;
  if (p.out_dtype == KVQ_OUT_F32) {
    float* o = reinterpret_cast<float*>(p.out) + orow;
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = acc[i];
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + orow;
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = __float2bfloat16_rn(acc[i]);
  }
}

template <int D>
int ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    const size_t sm = Smem<D>::bytes(64);
    cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(Smem<D>::bytes(4096)));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<D>, kThreads, sm) != cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int D>
cudaError_t launch_pair(const DParams& p, int C, int B, int Hq, cudaStream_t stream) {
  decode_split_kernel<D><<<C, kThreads, Smem<D>::bytes(B), stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the merge may start while the split grid drains (programmatic dependent launch);
  // it waits for the split grid's completion before reading the partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((B * Hq + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
}

}  // namespace

int decode_num_ctas(int D) {
  const int per = D == 128 ? ctas_per_sm<128>() : ctas_per_sm<64>();
  return device_sm_count() * per;
}

// workspace: [pre: B+1 int32, padded to 16 B][lse: slots*rep f32, padded][o: slots*rep*D f32]
static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int D, int num_ctas) {
  const size_t rep = static_cast<size_t>(Hq / Hkv);
  const size_t slots = static_cast<size_t>(B) * Hkv + num_ctas;
  return align16((B + 1) * 4) + align16(slots * rep * 4) + slots * rep * D * 4;
}

kvq_status launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const kvq_cache& K = *a.k;
  const kvq_cache& Vc = *a.v;
  const int D = K.D, B = K.B, Hkv = K.Hkv, Tcap = K.Tcap;
  if (B > 4096) return KVQ_ERR_UNSUPPORTED;  // dynamic shared memory was sized for B <= 4096
  const int C = decode_num_ctas(D);
  const size_t need = decode_workspace_bytes(B, a.Hq, Hkv, D, C);
  if (a.ws == nullptr || a.ws_bytes < need) return KVQ_ERR_WORKSPACE;

  DParams p;
  memset(&p, 0, sizeof(p));
  const HeadLayout& hl = a.layout;
  const uint64_t rows8 = static_cast<uint64_t>(hl.n8) * B * Tcap;
  const uint64_t rows4 = static_cast<uint64_t>(hl.n4) * B * Tcap;
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
  p.ws_pre = reinterpret_cast<int32_t*>(ws);
  p.ws_lse = reinterpret_cast<float*>(ws + align16((B + 1) * 4));
  p.ws_o = reinterpret_cast<float*>(ws + align16((B + 1) * 4) + align16(slots * rep * 4));
  p.out = a.out;
  p.status = a.status;
  p.out_dtype = a.out_dtype;
  p.B = B; p.Hq = a.Hq; p.Hkv = Hkv; p.Tcap = Tcap; p.rep = rep; p.num_ctas = C;
  const float scale = a.softmax_scale > 0.0f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  for (int h = 0; h < KVQ_MAX_HKV; ++h) {
    p.plane[h] = hl.plane_idx[h];
    p.bits[h] = hl.bits[h];
  }
  const cudaError_t e = D == 128 ? launch_pair<128>(p, C, B, a.Hq, stream) : launch_pair<64>(p, C, B, a.Hq, stream);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
