// combine.cu -- the row gather into packed rows and the WeightedRowSum combine.
//
// gllm pull request #91, "What changes", MoE gather: one row gather fills the
// packed activation buffer (row r holds the token of pair perm_pair[r]), and
// one WeightedRowSum adds each token's topK expert outputs onto the pre-filled
// shared-expert output: dst[i] += sum_j w[i,j] * src[rows[i,j]].  Each
// element of dst has a single writer that walks j upward, so the sum needs no
// atomic adds and does not depend on how the threads are scheduled.
//
// Here each thread owns 8 consecutive columns of one dst row (one 16-byte bf16
// vector): it widens dst to fp32, adds w[i][j] * src[rows[i][j]][c] for
// j = 0..k-1 in order with one fused multiply-add each, and rounds once to
// bf16 (round to nearest even).  Out-of-range row indices add nothing.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCombineThreads = 256;
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kCombineThreads)
    weighted_row_sum_kernel(uint16_t* __restrict__ dst, const float* __restrict__ src,
                            const int32_t* __restrict__ rows, const float* __restrict__ w, int32_t n, int32_t k,
                            int32_t cols, int32_t src_rows) {
  pdl_wait();
  const int32_t vec_per_row = cols / 8;
  const long long total = (long long)n * vec_per_row;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
       v += (long long)gridDim.x * blockDim.x) {
    const int32_t i = (int32_t)(v / vec_per_row), c = (int32_t)(v % vec_per_row) * 8;
    uint4 d = *reinterpret_cast<const uint4*>(dst + (size_t)i * cols + c);
    float acc[8] = {bf16lo(d.x), bf16hi(d.x), bf16lo(d.y), bf16hi(d.y),
                    bf16lo(d.z), bf16hi(d.z), bf16lo(d.w), bf16hi(d.w)};
    for (int j = 0; j < k; ++j) {
      const int32_t r = rows[(size_t)i * k + j];
      if (r < 0 || r >= src_rows) continue;
      const float wj = w[(size_t)i * k + j];
      const float4* sp = reinterpret_cast<const float4*>(src + (size_t)r * cols + c);
      const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
      acc[0] = __fmaf_rn(wj, s0.x, acc[0]);
      acc[1] = __fmaf_rn(wj, s0.y, acc[1]);
      acc[2] = __fmaf_rn(wj, s0.z, acc[2]);
      acc[3] = __fmaf_rn(wj, s0.w, acc[3]);
      acc[4] = __fmaf_rn(wj, s1.x, acc[4]);
      acc[5] = __fmaf_rn(wj, s1.y, acc[5]);
      acc[6] = __fmaf_rn(wj, s1.z, acc[6]);
      acc[7] = __fmaf_rn(wj, s1.w, acc[7]);
    }
    d.x = pack_bf16x2(acc[0], acc[1]);
    d.y = pack_bf16x2(acc[2], acc[3]);
    d.z = pack_bf16x2(acc[4], acc[5]);
    d.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(dst + (size_t)i * cols + c) = d;
  }
}

// One warp per token: x[t] is read once and written to the packed rows of
// its k pairs (Xp[inv[t*k + j]][:] = x[t][:], pairs with inv = -1 skipped).
// Token-major, so a token's row is read from memory once rather than once per
// pair: with x larger than L2 the row-major form read it k times from HBM.
// Each lane keeps four 16-byte vectors in flight.
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ inv, int32_t n, int32_t k, int32_t H,
                  int32_t R, uint16_t* __restrict__ Xp) {
  pdl_wait();
  constexpr int kU = 4;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  const int vecs = H / 8;
  for (long long t = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); t < n; t += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int v0 = lane; v0 < vecs; v0 += 32 * kU) {
      uint4 buf[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + 32 * u < vecs) buf[u] = __ldg(src + v0 + 32 * u);
      for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(inv + t * k + j);
        if (r < 0 || r >= R) continue;
        uint4* d = reinterpret_cast<uint4*>(Xp + (size_t)r * H);
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (v0 + 32 * u < vecs) d[v0 + 32 * u] = buf[u];
      }
    }
  }
  pdl_launch_dependents();
}

static int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

cudaError_t launch_weighted_row_sum(uint16_t* dst, const float* src, const int32_t* rows, const float* w,
                                    int32_t n, int32_t k, int32_t cols, int32_t src_rows, cudaStream_t s,
                                    bool pdl) {
  const long long total = (long long)n * (cols / 8);
  long long blocks = (total + kCombineThreads - 1) / kCombineThreads;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_ex(weighted_row_sum_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, s, pdl, dst, src,
                   rows, w, n, k, cols, src_rows);
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int32_t n, int32_t k, int32_t H, int32_t R,
                          uint16_t* Xp, cudaStream_t s, bool pdl) {
  long long blocks = ((long long)n + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_ex(gather_kernel, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, pdl, x, inv, n, k, H, R, Xp);
}

}  // namespace moe
