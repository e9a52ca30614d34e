// gemv.cu -- NVFP4 weight-streaming path for experts with few packed rows.
//
// gllm pull request #91, "Results": experts holding at most 32 tokens run an
// NVFP4 GEMV instead of the tensor-core GEMM; TensorFold issue #2265
// ("Proposal") measures the same kind of kernel as load-latency bound and keeps
// the k order of each row's sum fixed so every output bit stays the same.
//
// One launch covers every expert that takes this path.  A warp owns one
// weight row (expert e, output feature n) at a time and streams it straight
// from HBM with 128-bit loads, one 16-byte chunk (32 codes) per lane per step,
// the next row's chunks already in flight while the current one is summed.
// Codes are unpacked exactly to bf16 (a code-pair lookup times the e4m3 block
// scale; 2 + 4 significant bits fit in bf16's 8), multiplied against the
// bf16 activations with fp32 fused multiply-adds, and reduced across the warp
// with shuffles in a fixed butterfly order, so results are run-to-run
// identical.  relu^2 and the bf16 rounding of the up projection are fused
// into the store.  For a gated expert the warp streams the gate row and the
// up row of the same feature together and stores bf16(silu(gate) * up).
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kGemvTok = 4;         // tokens summed per pass over a weight row
constexpr int kGemvMaxChunks = 4;   // K <= 32 * 32 * 4 = 4096 per lane-chunk plan
constexpr int kMaxExperts = 1024;

// e2m1 magnitudes as bf16 bit patterns, codes 0..7 (0, 0.5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ uint32_t e2m1_bf16_bits(uint32_t code) {
  const uint32_t mag = code & 7u, e = mag >> 1, m = mag & 1u;
  uint32_t bits = 0;
  if (e == 0) bits = m ? 0x3F00u : 0u;                       // 0.5 or 0
  else bits = ((126u + e) << 7) | (m << 6);                  // 2^(e-1) * (1 + m/2)
  return bits | ((code & 8u) << 12);
}

// e4m3 (E4M3FN) byte -> bf16 value, exact (3 mantissa bits fit in bf16's 7).
__device__ __forceinline__ uint32_t e4m3_bf16_bits(uint32_t b) {
  const uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
  float v = (e == 0) ? (float)m * 0.001953125f /* 2^-9 */ : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (uint32_t)f2bf_rn(v) | (s << 15);
}

// d = a.lo * b.lo + d, then a.hi * b.hi + d: bf16 inputs, fp32 accumulate, one rounding each.
__device__ __forceinline__ void fma2_bf16(float& d, uint32_t a, uint32_t b) {
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %0, ah, bh, %0;\n}\n"
      : "+f"(d)
      : "r"(a), "r"(b));
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct RowChunks {
  uint4 c[kGemvMaxChunks];
  uint32_t s[kGemvMaxChunks];  // two scale bytes per chunk
};

__device__ __forceinline__ void load_row(RowChunks& r, const uint8_t* codes_row, const uint8_t* scales_row,
                                         int nchunks, int lane) {
#pragma unroll
  for (int i = 0; i < kGemvMaxChunks; ++i) {
    const int ch = lane + 32 * i;
    if (ch < nchunks) {
      r.c[i] = ldg_stream(codes_row + 16 * ch);
      r.s[i] = *reinterpret_cast<const uint16_t*>(scales_row + 2 * ch);
    }
  }
}

// One row's partial dot products against the pass's tokens (this lane's chunks).
__device__ __forceinline__ void row_dots(const RowChunks& rc, const uint32_t* lut_lane, const uint32_t* scale_lut,
                                         const uint16_t* const (&xrow)[kGemvTok], int nt, int nchunks, int lane,
                                         float (&acc)[kGemvTok]) {
#pragma unroll
  for (int i = 0; i < kGemvMaxChunks; ++i) {
    const int ch = lane + 32 * i;
    if (ch < nchunks) {
      const uint32_t s0 = scale_lut[rc.s[i] & 0xFFu], s1 = scale_lut[(rc.s[i] >> 8) & 0xFFu];
      const uint32_t words[4] = {rc.c[i].x, rc.c[i].y, rc.c[i].z, rc.c[i].w};
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t byte = (words[q] >> (8 * b)) & 0xFFu;
          w[4 * q + b] = hmul2_bf16(lut_lane[byte * 32], q < 2 ? s0 : s1);
        }
      }
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        if (t < nt) {
          const uint4* xp = reinterpret_cast<const uint4*>(xrow[t] + 32 * ch);
          uint4 xv[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) xv[v] = __ldg(xp + v);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            fma2_bf16(acc[t], w[4 * v + 0], xv[v].x);
            fma2_bf16(acc[t], w[4 * v + 1], xv[v].y);
            fma2_bf16(acc[t], w[4 * v + 2], xv[v].z);
            fma2_bf16(acc[t], w[4 * v + 3], xv[v].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kGemvTok; ++t) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], d);
  }
}

template <bool GATED>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(GemvArgs a) {
  __shared__ uint32_t lut[256 * 32];       // [code byte][lane]: bf16x2 (low nibble, high nibble)
  __shared__ uint32_t scale_lut[256];      // e4m3 byte -> bf16x2 (s, s)
  __shared__ int32_t act[kMaxExperts];
  __shared__ int32_t n_act_sm;
  __shared__ int32_t warp_cnt[kGemvWarps * 4];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 256 * 32; i += kGemvThreads) {
    const uint32_t byte = (uint32_t)i >> 5;
    lut[i] = e2m1_bf16_bits(byte & 15u) | (e2m1_bf16_bits(byte >> 4) << 16);
  }
  for (int i = tid; i < 256; i += kGemvThreads) {
    const uint32_t s = e4m3_bf16_bits((uint32_t)i);
    scale_lut[i] = s | (s << 16);
  }

  // Wait for the producer of counts / inputs before touching them.
  pdl_wait();

  // Compact list of the experts this path serves, in expert order.
  if (tid == 0) n_act_sm = 0;
  __syncthreads();
  for (int base = 0; base < a.E; base += kGemvThreads) {
    const int e = base + tid;
    bool mine = false;
    if (e < a.E) {
      const int c = a.counts[e];
      mine = c > 0 && (a.max_rows <= 0 || c <= a.max_rows);
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int before = n_act_sm;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    if (mine) act[before + __popc(bal & ((1u << lane) - 1u))] = e;
    __syncthreads();
    if (tid == 0) {
      int add = 0;
      for (int w = 0; w < kGemvWarps; ++w) add += warp_cnt[w];
      n_act_sm += add;
    }
    __syncthreads();
  }
  const int n_act = n_act_sm;
  pdl_launch_dependents();

  const int N = a.N, K = a.K, nchunks = K / 32;
  const size_t code_row = (size_t)K / 2, scale_row = (size_t)K / 16;
  const long long total = (long long)n_act * N;
  const long long gwarp = (long long)blockIdx.x * kGemvWarps + warp;
  const long long nwarps = (long long)gridDim.x * kGemvWarps;
  const uint32_t* lut_lane = lut + lane;

  RowChunks cur, nxt, gcur, gnxt;
  long long u = gwarp;
  if (u < total) {
    const int e = act[u / N], n = (int)(u % N);
    const size_t wr = (size_t)e * N + n;
    load_row(cur, a.codes + wr * code_row, a.scales + wr * scale_row, nchunks, lane);
    if (GATED) load_row(gcur, a.gate_codes + wr * code_row, a.gate_scales + wr * scale_row, nchunks, lane);
  }
  for (; u < total; u += nwarps) {
    const int e = act[u / N], n = (int)(u % N);
    const long long un = u + nwarps;
    if (un < total) {  // next row in flight while this one is summed
      const int e2 = act[un / N], n2 = (int)(un % N);
      const size_t wr = (size_t)e2 * N + n2;
      load_row(nxt, a.codes + wr * code_row, a.scales + wr * scale_row, nchunks, lane);
      if (GATED) load_row(gnxt, a.gate_codes + wr * code_row, a.gate_scales + wr * scale_row, nchunks, lane);
    }
    const int cnt = a.counts[e], off = a.offsets[e];
    const float g = a.global[e];
    for (int t0 = 0; t0 < cnt; t0 += kGemvTok) {
      const int nt = min(kGemvTok, cnt - t0);
      const uint16_t* xrow[kGemvTok];
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        const int r = off + t0 + min(t, nt - 1);
        const long long src = a.token_indexed ? (long long)(a.perm_pair[r] / a.k) : (long long)r;
        xrow[t] = a.in + (size_t)src * K;
      }
      float acc[kGemvTok], gacc[kGemvTok];
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) acc[t] = gacc[t] = 0.f;
      row_dots(cur, lut_lane, scale_lut, xrow, nt, nchunks, lane, acc);
      if (GATED) row_dots(gcur, lut_lane, scale_lut, xrow, nt, nchunks, lane, gacc);
      // lane t stores token t of this pass
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        if (lane == t && t < nt) {
          const size_t o = (size_t)(off + t0 + t) * N + n;
          const float h = g * acc[t];
          if (GATED) {
            const float gv = a.gate_global[e] * gacc[t];
            reinterpret_cast<uint16_t*>(a.out)[o] = f2bf_rn(gv / (1.0f + expf(-gv)) * h);
          } else if (a.relu2_bf16_out) {
            const float r = fmaxf(h, 0.f);
            reinterpret_cast<uint16_t*>(a.out)[o] = f2bf_rn(r * r);
          } else {
            reinterpret_cast<float*>(a.out)[o] = h;
          }
        }
      }
    }
    cur = nxt;
    if (GATED) gcur = gnxt;
  }
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms * 4;
  if (a.gate_codes) return launch_ex(gemv_kernel<true>, dim3(grid), dim3(kGemvThreads), 0, s, pdl, a);
  return launch_ex(gemv_kernel<false>, dim3(grid), dim3(kGemvThreads), 0, s, pdl, a);
}

}  // namespace moe
