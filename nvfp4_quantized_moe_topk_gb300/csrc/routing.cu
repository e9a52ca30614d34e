// routing.cu -- the permutation step of the MoE gather.
//
// gllm pull request #91 ("perf: gather tokens per MoE expert, run large NVFP4
// GEMMs on bf16 tensor cores"), section "What changes", MoE gather: every
// picked (token, expert) pair owns one row of an n*topK-row buffer whose rows
// are grouped by expert.  This kernel produces that permutation on the device:
//
//   counts[e]     rows of expert e
//   offsets[e]    exclusive prefix sum of counts (offsets[E] = kept rows)
//   perm_pair[r]  the pair p = t*k + j that owns packed row r
//   inv[p]        the packed row of pair p (-1 if its id is outside [0, E))
//
// Rows of one expert are in ascending pair order (a stable counting sort), so
// the result is unique and matches the oracle bit for bit.  One CTA of 1024
// threads: each warp owns a contiguous slice of the pairs; per-warp histograms
// in shared memory give every warp its starting row per expert; the warp then
// walks its slice 32 pairs at a time and ranks equal ids with __match_any_sync,
// which keeps pair order without any ordering atomics.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads, 1)
    routing_kernel(const int32_t* __restrict__ ids, int32_t R, int32_t E, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm_pair, int32_t* __restrict__ inv,
                   int32_t* __restrict__ err) {
  extern __shared__ int32_t sm_route[];
  int32_t* hist = sm_route;                      // [kRouteWarps][E]: count, then running row base
  int32_t* tot = sm_route + kRouteWarps * E;     // [E]
  int32_t* warp_sums = tot + E;                  // [kRouteWarps]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();

  const int32_t chunk = (R + kRouteWarps - 1) / kRouteWarps;
  const int32_t beg = min(R, warp * chunk), end = min(R, beg + chunk);
  int bad = 0;
  for (int32_t p = beg + lane; p < end; p += 32) {
    const int32_t e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&hist[warp * E + e], 1);
    else bad = 1;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kFlagBadRouting);
  __syncthreads();

  // totals per expert, then an exclusive scan over experts (E <= 1024)
  int32_t my_total = 0;
  if (tid < E) {
    for (int w = 0; w < kRouteWarps; ++w) my_total += hist[w * E + tid];
    tot[tid] = my_total;
  }
  // block-wide exclusive scan of my_total over tid
  int32_t incl = my_total;
  for (int d = 1; d < 32; d <<= 1) {
    int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t s = warp_sums[lane];
    for (int d = 1; d < 32; d <<= 1) {
      int32_t v = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += v;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int32_t excl = incl - my_total + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (tid < E) {
    counts[tid] = my_total;
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + my_total;
    // running base of each warp's slice for this expert
    int32_t base = excl;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int32_t c = hist[w * E + tid];
      hist[w * E + tid] = base;
      base += c;
    }
  }
  __syncthreads();

  // stable scatter: each warp walks its slice in order, 32 pairs per step
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int32_t p0 = beg; p0 < end; p0 += 32) {
    const int32_t p = p0 + lane;
    const bool live = p < end;
    const int32_t e = live ? ids[p] : -1;
    const bool valid = live && e >= 0 && e < E;
    const int32_t key = valid ? e : -1 - (int32_t)(!live);  // dropped / tail lanes never match valid ones
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int32_t r = -1;
    if (valid) r = hist[warp * E + e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
    if (live) {
      inv[p] = r;
      if (valid) perm_pair[r] = p;
    }
  }
}

size_t routing_smem_bytes(int E) { return sizeof(int32_t) * ((size_t)kRouteWarps * E + E + kRouteWarps); }

cudaError_t launch_routing(const int32_t* ids, int32_t R, int32_t E, int32_t* counts, int32_t* offsets,
                           int32_t* perm_pair, int32_t* inv, int32_t* err, cudaStream_t s) {
  const size_t smem = routing_smem_bytes(E);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(routing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  routing_kernel<<<1, kRouteThreads, smem, s>>>(ids, R, E, counts, offsets, perm_pair, inv, err);
  return cudaGetLastError();
}

}  // namespace moe
