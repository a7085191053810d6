// kvq_mask.cu -- a block-sparse tile mask for causal prefill, built on the GPU
// (《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 §2.3: whole tiles of
// the score matrix judged unnecessary are skipped, with the skipped share
// capped so that no block is starved; §1.3 for the mask's role).
//
// For query tile qt the candidates are the key tiles kt in [1, qt): strictly
// below the diagonal and not key tile 0.  Of its n = max(qt - 1, 0)
// candidates the row skips floor(n * num / den) (integer arithmetic, so the
// cap holds per row, exactly), namely those with the smallest keys
// SplitMix64(seed, qt * nT + kt + 1) -- output number qt * nT + kt + 1 of the
// SplitMix64 generator (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014) seeded with `seed` -- ties broken by the smaller
// kt.  Key tile 0 and the diagonal are always kept; tiles above the diagonal
// are 0 (causal prefill never reads them).
//
// One CTA per query tile: the candidates' (key, kt) pairs are sorted in
// shared memory by a bitonic network, then the first k are cleared.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kMaskThreads = 256;

// SplitMix64 output number `n` (1-based) of the generator seeded with `seed`:
// the state after n steps is seed + n * gamma, mixed by the generator's
// finaliser.
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t n) {
  uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(kMaskThreads) tile_mask_kernel(uint8_t* mask, int nT, int num, int den,
                                                                  uint64_t seed, int npow2) {
  extern __shared__ uint8_t smem_raw[];
  uint64_t* key = reinterpret_cast<uint64_t*>(smem_raw);
  uint16_t* idx = reinterpret_cast<uint16_t*>(key + npow2);
  const int qt = blockIdx.x;
  uint8_t* row = mask + static_cast<int64_t>(qt) * nT;
  const int n = qt > 1 ? qt - 1 : 0;
  const int k = static_cast<int>(static_cast<int64_t>(n) * num / den);
  for (int kt = threadIdx.x; kt < nT; kt += blockDim.x) row[kt] = kt <= qt ? 1 : 0;
  if (k == 0) return;
  // candidate j (0-based) is key tile j + 1; padding sorts last
  for (int j = threadIdx.x; j < npow2; j += blockDim.x) {
    if (j < n) {
      key[j] = splitmix64(seed, static_cast<uint64_t>(qt) * nT + (j + 1) + 1);
      idx[j] = static_cast<uint16_t>(j + 1);
    } else {
      key[j] = ~0ull;
      idx[j] = 0xFFFFu;
    }
  }
  __syncthreads();
  // bitonic sort of (key, idx) ascending over npow2 entries
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < npow2 / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));   // first index of the pair
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = key[lo], b = key[hi];
        const uint16_t ia = idx[lo], ib = idx[hi];
        const bool a_gt_b = a > b || (a == b && ia > ib);
        if (a_gt_b == up) {
          key[lo] = b; key[hi] = a;
          idx[lo] = ib; idx[hi] = ia;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x) row[idx[i]] = 0;
}

}  // namespace

cudaError_t launch_tile_mask(uint8_t* mask, int nT, int num, int den, uint64_t seed, cudaStream_t stream) {
  int npow2 = 1;
  while (npow2 < nT) npow2 <<= 1;
  const size_t smem = static_cast<size_t>(npow2) * (8 + 2);
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(tile_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  tile_mask_kernel<<<static_cast<unsigned>(nT), kMaskThreads, smem, stream>>>(mask, nT, num, den, seed, npow2);
  return cudaGetLastError();
}

}  // namespace kvq
