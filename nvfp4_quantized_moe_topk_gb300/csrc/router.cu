// router.cu -- top-k routing with softmax over the picked experts.
//
// The step before the layer: the layer's synthetic workloads are routed from
// fp32 logits (plus, for the prefill configurations, a per-expert bias added
// to them) by taking the top k and renormalising a softmax over the k picked;
// gllm pull request #91 ("What changes", MoE gather) then groups the picked
// (token, expert) pairs.  Here one warp routes one token:
//
//   z[e] = logits[t][e] + bias[e]        (one fp32 addition)
//   pick j = the best z among the experts not yet picked, in the order
//            (z descending, expert index ascending): a warp max over an
//            order-preserving integer key of z, then a warp min over the index
//   w[t][j] = exp(z_j - z_0) / sum_i exp(z_i - z_0)
//   counts[e] += 1 for every pick (optional fused histogram)
//
// Every selection is an exact fp32 comparison, so the ids equal any other
// evaluation of the same order bit for bit; the weights use expf and a sum in
// a fixed butterfly order, so they are run-to-run identical.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;          // warps per block
constexpr int kRouterMaxTokensPerWarp = 8;  // large batches: tokens routed by each warp in turn

// Unsigned key with the order of the fp32 value (after -0 -> +0, so that
// equal values compare equal as in the float comparison).
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t u = __float_as_uint(z + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Lane l's biased logits z[l + 32 i], i < SLOTS, of one token.
template <int SLOTS>
__device__ __forceinline__ void load_token(const float* __restrict__ row, const float* __restrict__ bias, int32_t E,
                                           int lane, float (&z)[SLOTS]) {
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int32_t e = lane + 32 * i;
    z[i] = 0.f;
    if (e < E) z[i] = bias ? __ldg(row + e) + __ldg(bias + e) : __ldg(row + e);
  }
}

// One warp routes one token from its loaded logits.  Each pick is the expert
// with the largest key among those not yet taken, equal keys taken lower index
// first (a max then a min over the warp).
template <int SLOTS>
__device__ __forceinline__ void route_token(const float (&z)[SLOTS], int32_t E, int32_t k, int lane,
                                            int32_t* __restrict__ ids_t, float* __restrict__ w_t, int32_t* s_hist) {
  uint32_t key[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) key[i] = lane + 32 * i < E ? order_key(z[i]) : 0u;  // 0: below every real key
  uint32_t taken = 0;
  float my_z = 0.f, z0 = 0.f;
  int32_t my_e = 0;
  for (int32_t j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int32_t be = 0x7fffffff;
    float bz = 0.f;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
      const int32_t e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && (be == 0x7fffffff || key[i] > bk)) {
        bk = key[i];
        be = e;
        bz = z[i];
      }
    }
    const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
    const int32_t ge = (int32_t)__reduce_min_sync(0xffffffffu, (be != 0x7fffffff && bk == gk) ? (uint32_t)be
                                                                                               : 0x7fffffffu);
    const float gz = __shfl_sync(0xffffffffu, bz, ge & 31);
    if ((ge & 31) == lane) taken |= 1u << (ge >> 5);
    if (j == 0) z0 = gz;
    if (lane == j) {
      my_z = gz;
      my_e = ge;
    }
  }
  const float ex = lane < k ? expf(my_z - z0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids_t[lane] = my_e;
    w_t[lane] = ex / sum;
    if (s_hist) atomicAdd(&s_hist[my_e], 1);
  }
}

template <int SLOTS>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int32_t n, int32_t E, int32_t k,
                  int32_t tpw, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts) {
  extern __shared__ int32_t s_hist[];  // [E] when counts are wanted
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (counts) {
    for (int32_t e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
  }
  const int64_t t0 = ((int64_t)blockIdx.x * kRouterWarps + warp) * tpw;
  float zc[SLOTS];
  if (t0 < n) load_token<SLOTS>(logits + t0 * E, bias, E, lane, zc);
  for (int32_t q = 0; q < tpw; ++q) {
    const int64_t t = t0 + q;
    if (t >= n) break;
    float zn[SLOTS];  // the next token's logits, in flight while this one is routed
    const bool more = q + 1 < tpw && t + 1 < n;
    if (more) load_token<SLOTS>(logits + (t + 1) * E, bias, E, lane, zn);
    route_token<SLOTS>(zc, E, k, lane, ids + t * k, w + t * k, counts ? s_hist : nullptr);
    if (more) {
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) zc[i] = zn[i];
    }
  }
  if (counts) {
    __syncthreads();
    if (gridDim.x == 1) {
      // one block routes every token: it writes the whole histogram (no
      // zeroing launch before it)
      for (int32_t e = threadIdx.x; e < E; e += blockDim.x) counts[e] = s_hist[e];
    } else {
      for (int32_t e = threadIdx.x; e < E; e += blockDim.x)
        if (s_hist[e]) atomicAdd(&counts[e], s_hist[e]);
    }
  }
}

template <int SLOTS>
cudaError_t launch_router_t(const float* logits, const float* bias, int32_t n, int32_t E, int32_t k, int32_t* ids,
                            float* w, int32_t* counts, cudaStream_t s) {
  // enough warps to hide a token's latency (~5k in flight), up to 8 tokens each
  // to cut the number of global histogram atomics on large batches (up to
  // kRouterWarps tokens make one block, which then writes the histogram itself)
  const int32_t tpw = (int32_t)std::max<long long>(1, std::min<long long>(kRouterMaxTokensPerWarp, n / 4864));
  const long long per_block = (long long)kRouterWarps * tpw;
  const long long blocks = ((long long)n + per_block - 1) / per_block;
  const size_t smem = counts ? (size_t)E * sizeof(int32_t) : 0;
  router_kernel<SLOTS><<<(unsigned)blocks, kRouterWarps * 32, smem, s>>>(logits, bias, n, E, k, tpw, ids, w, counts);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const float* logits, const float* bias, int32_t n, int32_t E, int32_t k, int32_t* ids,
                          float* w, int32_t* counts, cudaStream_t s) {
  const bool one_block = n > 0 && n <= kRouterWarps;
  if (counts && !one_block) {  // blocks add into counts: zero it first
    const cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
  }
  if (n == 0) return cudaSuccess;
  if (E <= 32) return launch_router_t<1>(logits, bias, n, E, k, ids, w, counts, s);
  if (E <= 64) return launch_router_t<2>(logits, bias, n, E, k, ids, w, counts, s);
  if (E <= 128) return launch_router_t<4>(logits, bias, n, E, k, ids, w, counts, s);
  if (E <= 256) return launch_router_t<8>(logits, bias, n, E, k, ids, w, counts, s);
  if (E <= 512) return launch_router_t<16>(logits, bias, n, E, k, ids, w, counts, s);
  if (E <= 1024) return launch_router_t<32>(logits, bias, n, E, k, ids, w, counts, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
