// kvq_prefill.cu -- prefill attention (causal or not) over the group-quantised KV cache
// on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Method (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》): the score matrix is
// cut into 128x128 tiles and never materialised; each tile's softmax statistics
// (running max, normaliser) are carried forward and a final correction divides
// by the normaliser (§2.2); whole key tiles may be skipped by a block-sparse
// mask (§1.3, §2.3); K and V are read as group-quantised codes and dequantised
// on the fly (§1.3, §2.4).  The attention itself is softmax(Q K^T / sqrt(d)) V
// (《一只"兔子"如何搅动大模型推理赛道的底层逻辑》 §3.1), with the causal rule or, for
// non-causal prefill, over every key of the sequence (then the mask may skip
// any off-diagonal tile; query tiles all carry nT key tiles).
//
// One CTA (512 threads, one per SM) computes one 128-row query tile for two
// query heads that share a KV head, so every dequantised K/V tile feeds two
// heads' products:
//   warp 0      allocates TMEM, loads the bf16 Q tiles by TMA, frees TMEM;
//   warp 1      one thread issues every tcgen05.mma:
//                 S_h = Q_h K^T (A, B from shared memory) and
//                 O_h += P_h V   (P from TMEM, V from shared memory);
//   warps 4-7   convert Q to fp16 in place, then per kept key tile read the
//               INT8 codes and fp16 scale/zero words from global memory and
//               write exact-rounded fp16 K_hat = (c - z) * s and V_hat tiles in
//               the 128-byte-swizzled layout the tensor core reads (2 stages);
//   warps 8-11  softmax of head 0, warps 12-15 softmax of head 1: one thread
//               per query row reads its S row from TMEM, applies the causal
//               rule on the diagonal tile (causal only), updates (max, sum) in the log2
//               domain, writes P (fp16) back over S, and at the end scales O by
//               1 / sum and stores it.
// TMEM (512 columns): S_0 [0,128) O_0 [128,256) S_1 [256,384) O_1 [384,512).
// The running max is only moved (and O rescaled) when it grows by more than
// 2^8, so P stays <= 256 and rescales are rare; the final division uses the
// sum accumulated against the same max, which keeps the result exact.
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kT = 128;           // tile edge (query rows, keys)
constexpr int kD = 128;           // head dim
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PParams {
  CUtensorMap tm_q;               // bf16 [B*Hq*S][128], box [64][128], 128B swizzle
  const uint8_t* kcodes;          // plane base of the K cache (all heads 8-bit)
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
};

// shared memory layout (bytes from a 1024-aligned base)
constexpr int kQBytes = kT * kD * 2;                 // one head, fp16: 32 KB (2 k-blocks of 16 KB)
constexpr int kOff_Q = 0;                            // 2 heads
constexpr int kOff_K = kOff_Q + 2 * kQBytes;         // 2 stages x 32 KB
constexpr int kOff_V = kOff_K + 2 * kQBytes;         // 2 stages x 32 KB
constexpr int kOff_Bar = kOff_V + 2 * kQBytes;
// barriers
enum {
  B_QFULL = 0, B_QREADY, B_KFULL0, B_KFULL1, B_VFULL0, B_VFULL1, B_KVEMPTY0, B_KVEMPTY1,
  B_SFULL0, B_SFULL1, B_PFULL0, B_PFULL1, B_ORDY0, B_ORDY1, B_DONE, B_COUNT
};
constexpr int kOff_Tmem = kOff_Bar + B_COUNT * 8;
constexpr int kSmemBytes = kOff_Tmem + 16 + 1024;

__device__ __forceinline__ bool tile_kept(const PParams& p, int qt, int kt) {
  return kt == qt || p.tile_mask == nullptr || p.tile_mask[qt * p.nT + kt] != 0;
}

// One 128-token x 128-channel code tile (K or V) of the dequant warpgroup,
// held in registers between its global loads and its conversion.  Thread wt
// (0..127), iteration it (0..7): k-block kb = it & 1 (64 channels), row
// 32 * (it >> 1) + 8 * (wt >> 5) + ((wt & 31) >> 2), 16 channels from
// chunk c8 = 4 * kb + (wt & 3).  A quarter warp then stores two adjacent rows,
// whose swizzled chunks never share banks.
struct CodeRegs {
  uint4 c[8];
  uint32_t sz[8];
};

__device__ __forceinline__ int dq_row(int it, int wt) { return 32 * (it >> 1) + 8 * (wt >> 5) + ((wt & 31) >> 2); }
__device__ __forceinline__ int dq_c8(int it, int wt) { return 4 * (it & 1) + (wt & 3); }

__device__ __forceinline__ void load_codes(CodeRegs& r, const uint8_t* codes, const uint32_t* sz, int wt) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = dq_row(it, wt), c8 = dq_c8(it, wt);
    r.c[it] = __ldg(reinterpret_cast<const uint4*>(codes + static_cast<size_t>(row) * kD + c8 * 16));
    r.sz[it] = __ldg(sz + row * 4 + (c8 >> 1));
  }
}

// fp16 K_hat / V_hat = (c - z) * s (exact difference, one rounding) into the
// 128-byte-swizzled K-major operand layout: [2 k-blocks][128 rows][128 B].
__device__ __forceinline__ void store_dequant(uint8_t* dst, const CodeRegs& r, int wt) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = dq_row(it, wt), c8 = dq_c8(it, wt);
    const uint32_t word = r.sz[it];
    const uint32_t zb = zero_biased2(word);
    const uint32_t s2 = (word & 0xFFFFu) | (word << 16);
    const __half2 sh = *reinterpret_cast<const __half2*>(&s2);
    uint32_t o[8];
    const uint32_t w[4] = {r.c[it].x, r.c[it].y, r.c[it].z, r.c[it].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo = hsub2_u32(bytes01_biased(w[i]), zb);
      uint32_t hi = hsub2_u32(bytes23_biased(w[i]), zb);
      __half2 x = __hmul2(*reinterpret_cast<__half2*>(&lo), sh);
      __half2 y = __hmul2(*reinterpret_cast<__half2*>(&hi), sh);
      o[2 * i] = *reinterpret_cast<uint32_t*>(&x);
      o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&y);
    }
    const int kb = c8 >> 2, ch2 = (c8 & 3) * 2, sw = row & 7;
    uint8_t* rowp = dst + kb * (kT * 128) + row * 128;
    *reinterpret_cast<uint4*>(rowp + ((ch2 ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(rowp + (((ch2 + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// key tiles [0, kt_end) of query tile qt can take part (L: the sequence's length)
__device__ __forceinline__ int key_tile_end(const PParams& p, int qt, int L) {
  return p.causal ? qt + 1 : (L + kT - 1) / kT;
}

__device__ __forceinline__ int next_kept(const PParams& p, int qt, int kt, int end) {
  while (kt < end && !tile_kept(p, qt, kt)) ++kt;
  return kt;
}

// Zeros in the output rows of this work item (a query tile past its sequence's end).
__device__ __forceinline__ void zero_out_tile(const PParams& p, int b, int h0, int nh, int qt) {
  const size_t row0 = (static_cast<size_t>(b) * p.Hq + h0) * p.S + static_cast<size_t>(qt) * kT;
  const int vec_per_row = kD * (p.out_dtype == KVQ_OUT_F32 ? 4 : 2) / 16;
  for (int h = 0; h < nh; ++h) {
    uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                           (row0 + static_cast<size_t>(h) * p.S) * kD *
                                               (p.out_dtype == KVQ_OUT_F32 ? 4 : 2));
    for (int i = threadIdx.x; i < kT * vec_per_row; i += kThreads) base[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOff_Bar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOff_Tmem);
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
  // the sequence's length: a query tile wholly past it writes zeros and ends
  // here, before any barrier or TMEM is set up (the decision is the CTA's own)
  int L = p.S;
  if (p.lens != nullptr) {
    L = p.lens[b];
    if (L < 0 || L > p.S) {
      if (threadIdx.x == 0 && qt == 0) report(p.status, KVQ_ERR_INVALID_ARG);
      L = min(max(L, 0), p.S);
    }
  }
  if (qt * kT >= L) {
    zero_out_tile(p, b, h0, nh, qt);
    return;
  }
  const int q_valid = min(kT, L - qt * kT);   // query rows of this tile inside the sequence

  if (threadIdx.x == 0) {
    mbar_init(&bar[B_QFULL], 1);
    mbar_init(&bar[B_QREADY], 4);
    mbar_init(&bar[B_KFULL0], 4); mbar_init(&bar[B_KFULL1], 4);
    mbar_init(&bar[B_VFULL0], 4); mbar_init(&bar[B_VFULL1], 4);
    mbar_init(&bar[B_KVEMPTY0], 1); mbar_init(&bar[B_KVEMPTY1], 1);
    mbar_init(&bar[B_SFULL0], 1); mbar_init(&bar[B_SFULL1], 1);
    mbar_init(&bar[B_PFULL0], 4); mbar_init(&bar[B_PFULL1], 4);
    mbar_init(&bar[B_ORDY0], 1); mbar_init(&bar[B_ORDY1], 1);
    mbar_init(&bar[B_DONE], 4 * nh);
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
  const int kt_end = key_tile_end(p, qt, L);
  int n_kept = 0;
  for (int kt = 0; kt < kt_end; ++kt) n_kept += tile_kept(p, qt, kt) ? 1 : 0;

  if (warp < 4) {
  tc::reg_dealloc<80>();
  if (warp == 0) {
    // ---------------- Q by TMA, then wait for the end and free TMEM ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[B_QFULL], nh * kQBytes);
      for (int h = 0; h < nh; ++h) {
        const int32_t y = ((b * p.Hq + h0 + h) * p.S) + qt * kT;
        tma_2d_g2s(smem + kOff_Q + h * kQBytes, &p.tm_q, 0, y, &bar[B_QFULL]);
        tma_2d_g2s(smem + kOff_Q + h * kQBytes + kT * 128, &p.tm_q, 64, y, &bar[B_QFULL]);
      }
    }
    __syncwarp();
    mbar_wait(&bar[B_DONE], 0, p.status);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
    return;
  }

  if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane != 0) return;
    const uint32_t id_qk = tc::idesc_f16_f32(kT, kT, false);
    const uint32_t id_pv = tc::idesc_f16_f32(kT, kD, true);
    const uint32_t q_base = smem_u32(smem + kOff_Q);
    const uint32_t k_base = smem_u32(smem + kOff_K);
    const uint32_t v_base = smem_u32(smem + kOff_V);
    if (!mbar_wait(&bar[B_QREADY], 0, p.status)) return;
    tc::fence_after_sync();
    auto issue_qk = [&](int h, int st) {
      const uint32_t qh = q_base + h * kQBytes;
      const uint32_t kh = k_base + st * kQBytes;
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint32_t off = (s >> 2) * (kT * 128) + (s & 3) * 32;
        tc::mma_ss(tmem + h * 256, tc::smem_desc_sw128(qh + off, 16, 1024), tc::smem_desc_sw128(kh + off, 16, 1024),
                   id_qk, s > 0);
      }
      tc::commit(&bar[B_SFULL0 + h]);
    };
    bool ok = true;
    for (int j = 0; j < n_kept && ok; ++j) {
      const int st = j & 1;
      if (j == 0) {
        ok = mbar_wait(&bar[B_KFULL0], 0, p.status);
        tc::fence_after_sync();
        for (int h = 0; h < nh; ++h) issue_qk(h, 0);
      }
      ok = ok && mbar_wait(&bar[B_VFULL0 + st], (j >> 1) & 1, p.status);
      tc::fence_after_sync();
      for (int h = 0; h < nh && ok; ++h) {
        ok = mbar_wait(&bar[B_PFULL0 + h], j & 1, p.status);
        tc::fence_after_sync();
        const uint32_t vs = v_base + st * kQBytes;
#pragma unroll
        for (int s = 0; s < kT / 16; ++s)
          tc::mma_ts(tmem + h * 256 + 128, tmem + h * 256 + s * 8, tc::smem_desc_sw128(vs + s * 2048, kT * 128, 1024),
                     id_pv, (j > 0 || s > 0) ? 1u : 0u);
        tc::commit(&bar[B_ORDY0 + h]);
        if (j + 1 < n_kept) {
          if (h == 0) {
            ok = ok && mbar_wait(&bar[B_KFULL0 + ((j + 1) & 1)], ((j + 1) >> 1) & 1, p.status);
            tc::fence_after_sync();
          }
          if (ok) issue_qk(h, (j + 1) & 1);
        }
      }
      tc::commit(&bar[B_KVEMPTY0 + st]);
    }
    return;
  }

  return;   // warps 2, 3: no role
  }

  if (warp < 8) {
    tc::reg_alloc<192>();
    // ---------------- dequant warpgroup ----------------
    const int wt = threadIdx.x - 128;
    if (!mbar_wait(&bar[B_QFULL], 0, p.status)) return;
    bool finite = true;
    for (int i = wt; i < nh * kQBytes / 16; i += 128) {
      uint4* ptr = reinterpret_cast<uint4*>(smem + kOff_Q) + i;
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
      *ptr = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (!finite) report(p.status, KVQ_ERR_NONFINITE);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_QREADY]);

    const size_t plane = static_cast<size_t>(kvh) * p.B * p.Tcap + static_cast<size_t>(b) * p.Tcap;
    const uint8_t* kcodes = p.kcodes + plane * kD;
    const uint8_t* vcodes = p.vcodes + plane * kD;
    const uint32_t* ksz = p.ksz + plane * 4;
    const uint32_t* vsz = p.vsz + plane * 4;
    // two register sets: while one part (K or V of a tile) is converted, the
    // next part's codes are already on their way from L2 / HBM.  Positions
    // past a shorter sequence's end within its last tile read as zeros: the
    // quantiser cleared them (codes and scale/zero words 0), so a masked score
    // (P = 0) never meets a non-finite V_hat in the P.V product.
    CodeRegs ra, rb;
    int kt = next_kept(p, qt, 0, kt_end);
    if (kt < kt_end) load_codes(ra, kcodes + static_cast<size_t>(kt) * kT * kD, ksz + kt * kT * 4, wt);
    for (int j = 0; kt < kt_end; ++j) {
      const int st = j & 1;
      const int kt_next = next_kept(p, qt, kt + 1, kt_end);
      load_codes(rb, vcodes + static_cast<size_t>(kt) * kT * kD, vsz + kt * kT * 4, wt);
      if (j >= 2 && !mbar_wait(&bar[B_KVEMPTY0 + st], ((j >> 1) - 1) & 1, p.status)) return;
      store_dequant(smem + kOff_K + st * kQBytes, ra, wt);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_KFULL0 + st]);
      if (kt_next < kt_end)
        load_codes(ra, kcodes + static_cast<size_t>(kt_next) * kT * kD, ksz + kt_next * kT * 4, wt);
      store_dequant(smem + kOff_V + st * kQBytes, rb, wt);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_VFULL0 + st]);
      kt = kt_next;
    }
    return;
  }

  // ---------------- softmax warpgroups ----------------
  tc::reg_dealloc<120>();
  const int h = (warp - 8) >> 2;            // head slot 0 or 1
  if (h >= nh) return;
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
      const int climit = min(kT, L - kt * kT);
      masked = climit < kT;
      lim = climit - 1;
    }
    ok = mbar_wait(&bar[B_SFULL0 + h], j & 1, p.status);
    tc::fence_after_sync();
    // pass 1: row max
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t v[32];
      tc::ld_32x32b_x32(s_addr + c * 32, v);
      tc::wait_ld();
      if (!masked) {
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(v[i]));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = (c * 32 + i > lim) ? mx : fmaxf(mx, __uint_as_float(v[i]));
      }
    }
    const float m_tile = mx * sl2;
    float m_use = m_run, alpha = 1.0f;
    if (m_run == -INFINITY || m_tile > m_run + kRescaleThreshold) {
      m_use = fmaxf(m_run, m_tile);
      alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_use);
      m_run = m_use;
    }
    // pass 2: P = 2^(S*scale_log2 - m) as fp16 pairs, written over the part of S
    // already read (columns 16c.. of P after S columns 32c.. were loaded)
    float psum = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t v[32];
      uint32_t pk[16];
      tc::ld_32x32b_x32(s_addr + c * 32, v);
      tc::wait_ld();
      if (!masked) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(v[i]), sl2, -m_use));
          const float p1 = fast_exp2(fmaf(__uint_as_float(v[i + 1]), sl2, -m_use));
          psum += p0 + p1;
          pk[i / 2] = pack_half2(p0, p1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = (c * 32 + i > lim) ? 0.0f : fast_exp2(fmaf(__uint_as_float(v[i]), sl2, -m_use));
          const float p1 = (c * 32 + i + 1 > lim) ? 0.0f : fast_exp2(fmaf(__uint_as_float(v[i + 1]), sl2, -m_use));
          psum += p0 + p1;
          pk[i / 2] = pack_half2(p0, p1);
        }
      }
      tc::st_32x32b_x16(s_addr + c * 16, pk);
    }
    l_run = l_run * alpha + psum;
    // rescale O (rare): needs the previous P.V product finished
    if (__any_sync(0xffffffffu, alpha != 1.0f) && j > 0) {
      ok = ok && mbar_wait(&bar[B_ORDY0 + h], (j - 1) & 1, p.status);
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::ld_32x32b_x32(o_addr + c * 32, v);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tc::st_32x32b_x32(o_addr + c * 32, v);
      }
    }
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_PFULL0 + h]);
    ++j;
  }
  // epilogue: O / l
  if (ok && n_kept > 0) ok = mbar_wait(&bar[B_ORDY0 + h], (n_kept - 1) & 1, p.status);
  tc::fence_after_sync();
  // rows past the sequence's end are written as zeros
  const float inv = (l_run > 0.0f && r < q_valid) ? 1.0f / l_run : 0.0f;
  const size_t orow = (static_cast<size_t>(b) * p.Hq + h0 + h) * p.S + static_cast<size_t>(qt) * kT + r;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tc::ld_32x32b_x32(o_addr + c * 32, v);
    tc::wait_ld();
    if (p.out_dtype == KVQ_OUT_F32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kD + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                           __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
    } else {
      uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kD + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(v[8 * i + 2 * e]) * inv,
                                                   __uint_as_float(v[8 * i + 2 * e + 1]) * inv);
          w[e] = *reinterpret_cast<uint32_t*>(&t);
        }
        o[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bar[B_DONE]);
}

// Per device, set once under a lock: the kernel's large dynamic shared memory
// limit, and whether it was built with the 128 registers per thread that the
// register split above assumes.  1 = ready, -1 = not usable, 0 = not yet set.
std::mutex g_prep_mu;
int g_prep[64] = {};

int prepare_prefill_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(g_prep_mu);
  if (g_prep[dev] == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, prefill_kernel) != cudaSuccess || fa.numRegs != 128) {
      g_prep[dev] = -2;   // unsupported build
    } else if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
               cudaSuccess) {
      return -1;          // a CUDA error; try again on the next call
    } else {
      g_prep[dev] = 1;
    }
  }
  return g_prep[dev];
}

}  // namespace

kvq_status launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PParams p;
  memset(&p, 0, sizeof(p));
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Hq * a.S;
  if (qrows >= (uint64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (encode_tensor_map_2d(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kD, qrows, kD * 2, 64, kT,
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
  const float scale = a.softmax_scale > 0.0f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(kD));
  p.scale_log2 = scale * 1.4426950408889634f;
  const int prep = prepare_prefill_on_current_device();
  if (prep == -2) return KVQ_ERR_UNSUPPORTED;
  if (prep != 1) return KVQ_ERR_CUDA;
  const int64_t items = static_cast<int64_t>(p.nT) * a.B * a.Hkv * p.pairs;
  if (items >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  prefill_kernel<<<static_cast<unsigned>(items), kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
