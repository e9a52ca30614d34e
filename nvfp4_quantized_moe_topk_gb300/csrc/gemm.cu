// gemm.cu -- NVFP4 grouped GEMM on the sm_103a tensor cores (tcgen05 + TMEM).
//
// gllm pull request #91 ("perf: gather tokens per MoE expert, run large NVFP4
// GEMMs on bf16 tensor cores"), section "What changes", bf16 NVFP4 GEMM: past
// the GEMV threshold the NVFP4 weight is unpacked to bf16 -- without rounding:
// an e2m1 value carries 2 significant bits and an e4m3 scale up to 4, so
// their product needs no more than bf16's 8 -- and fed to
// a bf16 tensor-core GEMM whose alpha carries the per-tensor global.  There
// the unpack is a separate kernel writing a bf16 copy to global memory and the
// GEMM is a library call; here both live in one persistent kernel and the
// bf16 weights only ever exist in shared memory:
//
//   warp 0      producer: per k-block a TMA tile of activations (128 rows x
//               64 bf16, 128-byte swizzle), a TMA tile of codes (256 rows x
//               32 bytes) and cp.async copies of the matching e4m3 scales
//   warp 1      one elected thread issues tcgen05.mma (M=128, N<=256, K=16,
//               bf16 x bf16 -> fp32 in tensor memory)
//   warp 2      allocates / frees the 512 tensor-memory columns
//   warp 3      builds the tile list
//   warps 4-7   epilogue: tcgen05.ld, alpha (the global), then either fp32
//               stores or relu^2 + bf16 rounding fused into the store
//   warps 8-15  unpack codes x scales -> bf16 into the swizzled K-major layout
//               the MMA reads, then fence to the async proxy
//
// Tiles are (group g, 128 rows of g, 256 output features); groups are the
// experts whose row count exceeds the GEMV threshold, rows are the packed rows
// offsets[g] .. offsets[g] + counts[g] (rows past a group's end belong to the
// next group or are zero-filled by TMA; their results are not stored).  Two
// accumulators in tensor memory let the epilogue of one tile overlap the
// mainloop of the next.  Every barrier wait is bounded in wall time; a wait
// that runs out sets the timeout flag and every role unwinds.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;    // activation + code + scale stages
constexpr int kBStages = 2;   // unpacked bf16 weight stages
constexpr int kGemmThreads = 512;
constexpr int kDequantWarps = 8;
constexpr int kDequantThreads = kDequantWarps * 32;
constexpr int kMaxGroups = 1024;

constexpr uint32_t kABytes = kBM * kBK * 2;        // 16 KB
constexpr uint32_t kCodeBytes = kBN * kBK / 2;     // 8 KB
constexpr uint32_t kScaleBytes = kBN * kBK / 16;   // 1 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;        // 32 KB
constexpr uint32_t kLutBytes = 256 * 32 * 4;       // 32 KB, one copy per lane

namespace lay {  // shared-memory layout, offsets from the 1024-aligned base
constexpr uint32_t a = 0;
constexpr uint32_t b = a + kStages * kABytes;
constexpr uint32_t codes = b + kBStages * kBBytes;
constexpr uint32_t scales = codes + kStages * kCodeBytes;
constexpr uint32_t lut = scales + kStages * kScaleBytes;
constexpr uint32_t scale_lut = lut + kLutBytes;
constexpr uint32_t nbars = 2 * kStages + 2 * kBStages + 4 + 1;
constexpr uint32_t bars = scale_lut + 256 * 4;
constexpr uint32_t misc = bars + nbars * 8;
constexpr uint32_t tile_start = misc + 64;                 // int32 [kMaxGroups + 1]
constexpr uint32_t group_id = tile_start + (kMaxGroups + 1) * 4;  // int32 [kMaxGroups]
constexpr uint32_t end = group_id + kMaxGroups * 4;
constexpr uint32_t alloc = end + 1024;                     // + alignment slack
}  // namespace lay

__device__ __forceinline__ uint32_t e2m1_bf16_bits_g(uint32_t code) {
  const uint32_t mag = code & 7u, e = mag >> 1, m = mag & 1u;
  uint32_t bits = (e == 0) ? (m ? 0x3F00u : 0u) : (((126u + e) << 7) | (m << 6));
  return bits | ((code & 8u) << 12);
}
__device__ __forceinline__ uint32_t e4m3_bf16_bits_g(uint32_t b) {
  const uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
  float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (uint32_t)f2bf_rn(v) | (s << 15);
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      if (err) atomicOr(err, kFlagTimeout);
      return false;
    }
  }
}

struct TileInfo {
  int32_t g, row0, rows, n0, ncols;
};

__device__ __forceinline__ TileInfo decode_tile(int32_t t, const int32_t* tile_start, const int32_t* group_id,
                                                int32_t ngroups, const GemmArgs& a, int32_t n_tiles) {
  int lo = 0, hi = ngroups - 1;  // last selected group whose first tile <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  const int32_t local = t - tile_start[lo];
  const int32_t mt = local / n_tiles, nt = local % n_tiles;
  ti.g = group_id[lo];
  if (a.counts) {
    ti.row0 = a.offsets[ti.g] + mt * kBM;
    ti.rows = min(kBM, a.counts[ti.g] - mt * kBM);
  } else {
    ti.row0 = mt * kBM;
    ti.rows = min(kBM, a.M - mt * kBM);
  }
  ti.n0 = nt * kBN;
  ti.ncols = min(kBN, a.N - ti.n0);
  return ti;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay::bars);
  uint64_t* full_l = bars;                    // [kStages]  TMA tx + 32 cp.async arrivals
  uint64_t* empty_l = full_l + kStages;       // [kStages]  MMA commit
  uint64_t* full_b = empty_l + kStages;       // [kBStages] one arrival per dequant warp
  uint64_t* empty_b = full_b + kBStages;      // [kBStages] MMA commit
  uint64_t* tmem_full = empty_b + kBStages;   // [2]        MMA commit
  uint64_t* tmem_empty = tmem_full + 2;       // [2]        128 epilogue threads
  uint64_t* drain = tmem_empty + 2;           // [1]        final MMA commit
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + lay::misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + lay::misc + 8);
  int32_t* ngroups_sm = reinterpret_cast<int32_t*>(sm + lay::misc + 16);
  int32_t* total_sm = reinterpret_cast<int32_t*>(sm + lay::misc + 20);
  int32_t* tile_start = reinterpret_cast<int32_t*>(sm + lay::tile_start);
  int32_t* group_id = reinterpret_cast<int32_t*>(sm + lay::group_id);
  uint32_t* lut = reinterpret_cast<uint32_t*>(sm + lay::lut);
  uint32_t* scale_lut = reinterpret_cast<uint32_t*>(sm + lay::scale_lut);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- set-up
  for (int i = tid; i < 256 * 32; i += kGemmThreads) {
    const uint32_t byte = (uint32_t)i >> 5;
    lut[i] = e2m1_bf16_bits_g(byte & 15u) | (e2m1_bf16_bits_g(byte >> 4) << 16);
  }
  for (int i = tid; i < 256; i += kGemmThreads) {
    const uint32_t s = e4m3_bf16_bits_g((uint32_t)i);
    scale_lut[i] = s | (s << 16);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_l[s], 1 + 32);
      mbar_init(&empty_l[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&full_b[s], kDequantWarps);
      mbar_init(&empty_b[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }

  // Inputs (counts, packed activations) come from the previous kernel.
  pdl_wait();

  const int32_t n_tiles = (a.N + kBN - 1) / kBN;
  if (warp == 3) {  // tile list: selected groups in order, n-tiles fastest
    if (a.counts == nullptr) {
      if (lane == 0) {
        tile_start[0] = 0;
        group_id[0] = 0;
        *ngroups_sm = a.M > 0 ? 1 : 0;
        *total_sm = ((a.M + kBM - 1) / kBM) * n_tiles;
      }
    } else {
      int32_t run = 0, ng = 0;
      for (int base = 0; base < a.G; base += 32) {
        const int g = base + lane;
        int32_t tiles = 0;
        bool sel = false;
        if (g < a.G) {
          const int32_t c = a.counts[g];
          sel = c > 0 && c > a.min_rows;
          if (sel) tiles = ((c + kBM - 1) / kBM) * n_tiles;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, sel);
        int32_t incl = tiles;
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += v;
        }
        if (sel) {
          const int slot = ng + __popc(bal & ((1u << lane) - 1u));
          tile_start[slot] = run + incl - tiles;
          group_id[slot] = g;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
        ng += __popc(bal);
      }
      if (lane == 0) {
        *ngroups_sm = ng;
        *total_sm = run;
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t ngroups = *ngroups_sm, total_tiles = *total_sm;
  pdl_launch_dependents();

  const int32_t kblocks = a.K / kBK;
  const size_t scale_row = (size_t)a.K / 16;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t outstanding = 0;          // stages whose last fill may still be landing
    uint32_t issued_phase[kStages] = {};
    bool ok = true;
    for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile(t, tile_start, group_id, ngroups, a, n_tiles);
      const int32_t wrow0 = ti.g * a.N + ti.n0;  // first weight row of the tile
      const uint8_t* srow = a.scales + (size_t)wrow0 * scale_row;
      for (int32_t kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&empty_l[stage], phase ^ 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        // the previous fill of this stage was consumed, so it has landed
        if (lane == 0) {
          mbar_arrive_expect_tx(&full_l[stage], kABytes + kCodeBytes);
          tma_load_2d(sm + lay::a + stage * kABytes, &tmA, kb * kBK, ti.row0, &full_l[stage]);
          tma_load_2d(sm + lay::codes + stage * kCodeBytes, &tmB, kb * (kBK / 2), wrow0, &full_l[stage]);
        }
        uint8_t* sscale = sm + lay::scales + stage * kScaleBytes;
        for (int r = lane; r < ti.ncols; r += 32) cp_async4(sscale + 4 * r, srow + (size_t)r * scale_row + 4 * kb);
        cp_async_arrive_noinc(&full_l[stage]);
        outstanding |= 1u << stage;
        issued_phase[stage] = phase;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      // Unwinding: let every copy this warp issued land before the CTA exits
      // (bounded: 1 ms per stage).
      asm volatile("cp.async.wait_all;" ::: "memory");
      for (int s = 0; s < kStages; ++s) {
        if (!(outstanding & (1u << s))) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full_l[s], issued_phase[s]) && globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0, bstage = 0, it = 0;
    uint32_t phase = 0, bphase = 0;
    bool ok = true;
    for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(t, tile_start, group_id, ngroups, a, n_tiles);
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      if (!wait_bar(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, a.err)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kBM, (uint32_t)ti.ncols);
      const uint32_t d_tmem = tmem_base + acc * kBN;
      for (int32_t kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&full_l[stage], phase, abort_flag, a.err) ||
            !wait_bar(&full_b[bstage], bphase, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_base = smem_u32(sm + lay::a + stage * kABytes);
          const uint32_t b_base = smem_u32(sm + lay::b + bstage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_bf16(d_tmem, smem_desc_k128(a_base + kk * 32), smem_desc_k128(b_base + kk * 32), idesc,
                        (kb | kk) != 0);
          }
          tc_commit(&empty_l[stage]);
          tc_commit(&empty_b[bstage]);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++bstage == kBStages) {
          bstage = 0;
          bphase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&tmem_full[acc]);
      __syncwarp();
    }
    // all MMAs this thread issued have completed once `drain` flips
    if (lane == 0) tc_commit(drain);
    __syncwarp();
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
    const int m = 32 * q + lane;
    int it = 0;
    for (int32_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(t, tile_start, group_id, ngroups, a, n_tiles);
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      if (!wait_bar(&tmem_full[acc], acc_phase, abort_flag, a.err)) break;
      tc_fence_after();
      const float alpha = a.global ? a.global[ti.g] : a.alpha0;
      const bool live = m < ti.rows;
      const size_t orow = (size_t)(ti.row0 + m) * a.N + ti.n0;
      for (int c = 0; c < ti.ncols; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + acc * kBN + c, r);
        tmem_ld_wait();
        if (live) {
          if (a.epilogue == 1) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float h0 = fmaxf(alpha * __uint_as_float(r[2 * i]), 0.f);
              const float h1 = fmaxf(alpha * __uint_as_float(r[2 * i + 1]), 0.f);
              o[i] = pack_bf16x2(h0 * h0, h1 * h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + c);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + orow + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_float4(alpha * __uint_as_float(r[4 * i]), alpha * __uint_as_float(r[4 * i + 1]),
                                   alpha * __uint_as_float(r[4 * i + 2]), alpha * __uint_as_float(r[4 * i + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty[acc]);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ unpack
    const int dt = tid - 8 * 32;  // 0 .. 255
    const uint32_t* lut_lane = lut + lane;
    int stage = 0, bstage = 0;
    uint32_t phase = 0, bphase = 0;
    bool ok = true;
    for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      for (int32_t kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&full_l[stage], phase, abort_flag, a.err) ||
            !wait_bar(&empty_b[bstage], bphase ^ 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint8_t* scodes = sm + lay::codes + stage * kCodeBytes;
        const uint8_t* sscale = sm + lay::scales + stage * kScaleBytes;
        uint8_t* sb = sm + lay::b + bstage * kBBytes;
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          const int item = dt + rep * kDequantThreads;  // (row n, half h) = (item / 2, item % 2)
          const int n = item >> 1, h = item & 1;
          const uint4 cw = *reinterpret_cast<const uint4*>(scodes + 32 * n + 16 * h);
          const uint32_t sc = *reinterpret_cast<const uint16_t*>(sscale + 4 * n + 2 * h);
          const uint32_t s0 = scale_lut[sc & 0xFFu], s1 = scale_lut[sc >> 8];
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
          uint32_t w[16];
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              const uint32_t byte = (words[qd] >> (8 * bb)) & 0xFFu;
              w[4 * qd + bb] = bf16x2_mul(lut_lane[byte * 32], qd < 2 ? s0 : s1);
            }
          }
          uint8_t* row = sb + 128 * n;
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            const int chunk = (4 * h + qd) ^ (n & 7);
            *reinterpret_cast<uint4*>(row + 16 * chunk) =
                make_uint4(w[4 * qd + 0], w[4 * qd + 1], w[4 * qd + 2], w[4 * qd + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_b[bstage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++bstage == kBStages) {
          bstage = 0;
          bphase ^= 1u;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int num_sms,
                        cudaStream_t s, bool pdl) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = raise_smem_limit(nvfp4_gemm_kernel, (int)lay::alloc, configured);
  if (e != cudaSuccess) return e;
  int grid = num_sms;
  if (a.counts == nullptr) {
    const long long tiles = (long long)((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
    if (tiles < grid) grid = (int)tiles;
  }
  if (grid < 1) grid = 1;
  return launch_ex(nvfp4_gemm_kernel, dim3(grid), dim3(kGemmThreads), lay::alloc, s, pdl, tmA, tmB, a);
}

// ------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

cudaError_t make_tmap_act(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K) {
  return make_tmap_act_rows(map, base, rows, K, kBM);
}

cudaError_t make_tmap_act_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_codes(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {K / 2, rows};
  const cuuint64_t strides[1] = {K / 2};
  const cuuint32_t box[2] = {kBK / 2, kBN};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace moe
