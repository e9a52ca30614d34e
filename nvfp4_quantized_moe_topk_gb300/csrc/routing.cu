// routing.cu -- the permutation step of the MoE gather.
//
// gllm pull request #91 ("perf: gather tokens per MoE expert, run large NVFP4
// GEMMs on bf16 tensor cores"), section "What changes", MoE gather: every
// picked (token, expert) pair owns one row of an n*topK-row buffer whose rows
// are grouped by expert.  These kernels produce that permutation on the device:
//
//   counts[e]     rows of expert e
//   offsets[e]    exclusive prefix sum of counts (offsets[E] = kept rows)
//   perm_pair[r]  the pair p = t*k + j that owns packed row r
//   inv[p]        the packed row of pair p (-1 if its id is outside [0, E))
//
// Rows of one expert are in ascending pair order (a stable counting sort), so
// the result is unique and matches the oracle bit for bit.
//
// The pairs are cut into slices of kSlice; one CTA of 1024 threads owns a
// slice.  With more than one slice a first kernel writes each slice's
// per-expert histogram, and the scatter kernel of slice b starts expert e's
// rows at offsets[e] + (rows of e in slices before b).  Inside a slice each
// warp owns a contiguous run of pairs; per-warp histograms in shared memory
// give every warp its starting row per expert; the warp then walks its run 32
// pairs at a time and ranks equal ids with __match_any_sync, which keeps pair
// order without any ordering atomics.  A batch of one slice needs the scatter
// kernel alone.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Histogram of slice b into blk_hist[b][0..E); flags ids outside [0, E).
__global__ void __launch_bounds__(kRouteThreads, 1)
    routing_hist_kernel(const int32_t* __restrict__ ids, int32_t R, int32_t E, int32_t* __restrict__ blk_hist,
                        int32_t* __restrict__ err) {
  extern __shared__ int32_t sm_hist[];  // [E]
  const int tid = threadIdx.x;
  for (int i = tid; i < E; i += kRouteThreads) sm_hist[i] = 0;
  __syncthreads();
  const int64_t beg = (int64_t)blockIdx.x * kRoutingSlice;
  const int64_t end = beg + kRoutingSlice < R ? beg + kRoutingSlice : R;
  int32_t e_reg[kRoutingSlice / kRouteThreads];
#pragma unroll
  for (int j = 0; j < kRoutingSlice / kRouteThreads; ++j) {  // all loads in flight first
    const int64_t p = beg + tid + (int64_t)j * kRouteThreads;
    e_reg[j] = p < end ? ids[p] : 0;
  }
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kRoutingSlice / kRouteThreads; ++j) {
    const int64_t p = beg + tid + (int64_t)j * kRouteThreads;
    if (p < end) {
      const int32_t e = e_reg[j];
      if (e >= 0 && e < E) atomicAdd(&sm_hist[e], 1);
      else bad = true;
    }
  }
  if (bad) atomicOr(err, kFlagBadRouting);
  pdl_launch_dependents();
  __syncthreads();
  for (int i = tid; i < E; i += kRouteThreads) blk_hist[(int64_t)blockIdx.x * E + i] = sm_hist[i];
}

// Counts, offsets and the stable scatter of slice b.  blk_hist (nullptr for
// a single slice) holds the G slices' histograms from routing_hist_kernel.
__global__ void __launch_bounds__(kRouteThreads, 1)
    routing_kernel(const int32_t* __restrict__ ids, int32_t R, int32_t E, const int32_t* __restrict__ blk_hist,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm_pair,
                   int32_t* __restrict__ inv, int32_t* __restrict__ err) {
  extern __shared__ int32_t sm_route[];
  int32_t* hist = sm_route;                      // [kRouteWarps][E]: count, then running row base
  int32_t* warp_sums = sm_route + kRouteWarps * E;  // [kRouteWarps]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();

  const int32_t sbeg = (int32_t)((int64_t)blockIdx.x * kRoutingSlice);
  const int32_t send = sbeg + kRoutingSlice < R ? sbeg + kRoutingSlice : R;
  const int32_t chunk = (send - sbeg + kRouteWarps - 1) / kRouteWarps;
  const int32_t beg = min(send, sbeg + warp * chunk), end = min(send, beg + chunk);
  int bad = 0;
  for (int32_t p = beg + lane; p < end; p += 32) {
    const int32_t e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&hist[warp * E + e], 1);
    else bad = 1;
  }
  if (!blk_hist && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kFlagBadRouting);
  __syncthreads();

  // per expert (tid < E, E <= 1024): this slice's count, the rows of the
  // slices before it, and the total over all slices
  int32_t mine = 0, before = 0, total = 0;
  if (tid < E) {
    for (int w = 0; w < kRouteWarps; ++w) mine += hist[w * E + tid];
    total = mine;
  }
  if (blk_hist) {
    pdl_wait();  // the histograms come from the previous kernel
    if (tid < E) {
      total = 0;
      for (int32_t b = 0; b < (int32_t)gridDim.x; ++b) {
        const int32_t v = blk_hist[(int64_t)b * E + tid];
        total += v;
        before += b < (int32_t)blockIdx.x ? v : 0;
      }
    }
  }
  // block-wide exclusive scan of total over tid
  int32_t incl = total;
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
  const int32_t excl = incl - total + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (tid < E) {
    if (blockIdx.x == 0) {
      counts[tid] = total;
      offsets[tid] = excl;
      if (tid == E - 1) offsets[E] = excl + total;
    }
    // running base of each warp's run for this expert
    int32_t base = excl + before;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int32_t c = hist[w * E + tid];
      hist[w * E + tid] = base;
      base += c;
    }
  }
  __syncthreads();

  // stable scatter: each warp walks its run in order, 32 pairs per step
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

size_t routing_smem_bytes(int E) { return sizeof(int32_t) * ((size_t)kRouteWarps * E + kRouteWarps); }

size_t routing_scratch_ints(int64_t R, int E) {
  const int64_t G = (R + kRoutingSlice - 1) / kRoutingSlice;
  return G > 1 ? (size_t)(G * E) : 0;
}

cudaError_t launch_routing(const int32_t* ids, int32_t R, int32_t E, int32_t* counts, int32_t* offsets,
                           int32_t* perm_pair, int32_t* inv, int32_t* err, cudaStream_t s, int32_t* blk_hist) {
  const size_t smem = routing_smem_bytes(E);
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = raise_smem_limit(routing_kernel, 200 * 1024, configured);
  if (e != cudaSuccess) return e;
  const int64_t G = ((int64_t)R + kRoutingSlice - 1) / kRoutingSlice;
  if (G <= 1 || !blk_hist) {
    if (G > 1) return cudaErrorInvalidValue;  // several slices need the histogram scratch
    routing_kernel<<<1, kRouteThreads, smem, s>>>(ids, R, E, nullptr, counts, offsets, perm_pair, inv, err);
    return cudaGetLastError();
  }
  routing_hist_kernel<<<(unsigned)G, kRouteThreads, (size_t)E * sizeof(int32_t), s>>>(ids, R, E, blk_hist, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_ex(routing_kernel, dim3((unsigned)G), dim3(kRouteThreads), smem, s, true, ids, R, E,
                   (const int32_t*)blk_hist, counts, offsets, perm_pair, inv, err);
}

}  // namespace moe
