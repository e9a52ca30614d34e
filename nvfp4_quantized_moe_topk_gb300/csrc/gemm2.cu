// gemm2.cu -- grouped NVFP4 GEMM for the layer, weights as the tensor-memory operand.
//
// gllm pull request #91 ("What changes", bf16 NVFP4 GEMM): above the GEMV
// threshold the NVFP4 weight is unpacked to bf16 -- without rounding, because
// an e2m1 value (2 significant bits) times an e4m3 scale (up to 4) needs no
// more than bf16's 8 -- and multiplied on
// bf16 tensor cores, with the per-tensor global in the GEMM's alpha.  On sm_103a
// the unpacked weight never needs to touch shared memory: tcgen05.mma can read
// its A operand from tensor memory, so the unpack warps write the bf16 weights
// straight from registers into TMEM (tcgen05.st) and only the activation tile
// travels through shared memory.  Per 64-wide k-block of a 128-feature x
// 224-token tile that is 28 KB of activations written by TMA and read by the
// MMA plus 4.5 KB of packed weights, against 448 cycles of MMA work.
//
// The time per k-block is nearly independent of the tile's token count (the
// unpack and the single issuing thread cost the same for any N), so the
// kernel runs as few, wide token tiles as tensor memory allows: two
// accumulators of 224 columns leave 64 columns for the unpacked weights.
// Measured against 192-token tiles with four A stages: 10-11% faster on both
// projections; 176-token tiles with five A stages were 8-10% slower.
//
//   D[feature][token] = sum_k W[feature][k] * X[token][k]   (M = 128 features,
//   N = tokens of the tile rounded up to 16, at most 224; K-major operands)
//
//   warp 0      producer: per k-block one 1-D bulk copy of the packed weight
//               block (128 rows x 32 code bytes + 128 x 4 scale bytes) and one
//               TMA tile of activations (224 rows x 64 bf16, 128-byte swizzle)
//   warp 1      one thread issues tcgen05.mma.cta_group::1.kind::f16 with A
//               in TMEM, B in shared memory, D in TMEM (two accumulators)
//   warp 2      allocates / frees the 512 TMEM columns; waits on the stage
//               barriers for the issuer and hands each k-block over through a
//               named barrier (the issuer must not read shared memory)
//   warp 3      builds the tile list (experts above the threshold)
//   warps 4-19  unpack, in two groups of 8 taking alternate k-blocks: thread =
//               (feature row, half of the k-block); 16 code bytes -> 16 bf16
//               pairs (bit placement + one bf16 multiply by the scale),
//               tcgen05.st into the A stage of its TMEM lane (group g always
//               fills stage g); a warp signals the stage ready as soon as its
//               store has landed (the A stages are the tightest buffer between
//               unpack and MMA: waiting one more k-block to hide the store's
//               latency measured 3% slower)
//   warps 20-23 epilogue: tcgen05.ld, alpha, fp32 rows or bf16(relu^2) rows;
//               for a gated expert the weight rows come in groups of 16 gate
//               rows then the 16 up rows of the same features, so TMEM lanes
//               l and l + 16 of a warp meet in one shuffle per two token
//               columns and store bf16(silu(gate) * up)
//
// TMEM columns: accumulators [0,224) and [224,448), two 32-column A stages
// from 448.  Tiles are (expert, 224 packed rows, 128 features), features
// fastest.  Every wait is bounded in wall time; a wait that runs out sets the
// timeout flag and every role unwinds.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace g2 {
constexpr int kM = 128;        // features per tile
constexpr int kN = kGemmTileRows;  // packed rows (tokens) per tile
constexpr int kK = 64;
constexpr int kWStages = 8;    // packed weight blocks (shared memory)
constexpr int kBStages = 6;    // activation tiles (shared memory): ~2.7k cycles of MMA work in flight
constexpr int kAStages = 2;    // unpacked weights (tensor memory)
constexpr int kUnpackWarps = 8;      // per group (one k-block: 4 row quarters x 2 halves)
constexpr int kUnpackGroups = 2;
constexpr int kThreads = 32 * (4 + kUnpackGroups * kUnpackWarps + 4);
constexpr int kMaxGroups = 1024;
constexpr uint32_t kWBytes = kGemmBlockBytes;     // 4608
constexpr uint32_t kBBytes = kN * kK * 2;         // 28 KB
constexpr uint32_t kAccCols = kN;                  // fp32 columns per accumulator
constexpr uint32_t kACol0 = 2 * kAccCols;          // first A-stage column
constexpr uint32_t kAStageCols = kK / 2;           // 32 columns of bf16 pairs

// shared-memory layout, offsets from the 1024-aligned base
constexpr uint32_t b = 0;
constexpr uint32_t w = b + kBStages * kBBytes;
constexpr uint32_t scale_lut = w + kWStages * kWBytes;
constexpr uint32_t nbars = 2 * kWStages + 2 * kBStages + 2 * kAStages + 4 + 1;
constexpr uint32_t bars = scale_lut + 256 * 4;
constexpr uint32_t misc = bars + nbars * 8;
constexpr uint32_t tile_start = misc + 64;
constexpr uint32_t group_id = tile_start + (kMaxGroups + 1) * 4;
constexpr uint32_t part_start = group_id + kMaxGroups * 4;
constexpr uint32_t end = part_start + (kMaxGroups + 1) * 4;
constexpr uint32_t alloc = end + 1024;
}  // namespace g2

// ------------------------------------------------------------------ repack
// Packed weight block (e, rb, kb): 128 rows x 8 words of bit-placed codes (the
// word layout of the streaming kernel: unpack_word yields the pairs k 0-1,
// 2-3, 4-5, 6-7 of the word), the two 16-byte halves of a row swapped on rows
// with bit 2 set so that 8 consecutive rows read one half on distinct banks;
// then 128 rows x 4 e4m3 scale bytes.  Rows past N are zero.
__global__ void repack_gemm_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                   int32_t G, int32_t N, int32_t K, uint8_t* __restrict__ out) {
  const int32_t KB = K / 64, NB = (N + 127) / 128;
  const long long rows_total = (long long)G * NB * KB * 128;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < rows_total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i & 127);
    const long long blk = i >> 7;
    const int kb = (int)(blk % KB);
    const long long rest = blk / KB;
    const int rb = (int)(rest % NB);
    const long long grp = rest / NB;
    const int n = rb * 128 + r;
    uint8_t* ob = out + blk * kGemmBlockBytes;
    uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t sc = 0;
    if (n < N) {
      const uint8_t* src = codes + (grp * N + n) * (long long)(K / 2) + kb * 32;
#pragma unroll
      for (int wd = 0; wd < 8; ++wd) {
        uint32_t v = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t byte = src[4 * wd + p];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t code = (byte >> (4 * h)) & 15u;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) v |= ((code >> bb) & 1u) << code_bit_pos(p, h, bb);
          }
        }
        words[wd] = v;
      }
      const uint8_t* ss = scales + (grp * N + n) * (long long)(K / 16) + kb * 4;
      sc = (uint32_t)ss[0] | ((uint32_t)ss[1] << 8) | ((uint32_t)ss[2] << 16) | ((uint32_t)ss[3] << 24);
    }
    const int swap = (r >> 2) & 1;
    uint32_t* orow = reinterpret_cast<uint32_t*>(ob + r * 32);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int q = 0; q < 4; ++q) orow[4 * (hf ^ swap) + q] = words[4 * hf + q];
    *reinterpret_cast<uint32_t*>(ob + 4096 + r * 4) = sc;
  }
}

cudaError_t launch_repack_gemm(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                               uint8_t* out, cudaStream_t s) {
  const long long work = (long long)G * ((N + 127) / 128) * (K / 64) * 128;
  long long blocks = (work + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  if (blocks < 1) blocks = 1;
  repack_gemm_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, scales, G, N, K, out);
  return cudaGetLastError();
}

size_t gemm_blocks_bytes(int32_t G, int32_t N, int32_t K) {
  return (size_t)G * ((N + 127) / 128) * (K / 64) * kGemmBlockBytes;
}

// ------------------------------------------------------------------ helpers
namespace {

// 32 lanes x 32 bit, 16 consecutive columns from 16 registers per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulator).
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

}  // namespace

// ------------------------------------------------------------------ kernel
namespace {

struct G2Tile {
  int32_t g, row0, rows, n0;
};

// Tile t: the full token tiles of every selected group come first (t < n_full,
// group order, feature blocks fastest), then each group's last, partial token
// tile.  A partial tile costs less than a full one, so the round-robin over
// CTAs leaves the cheap tiles for the last rounds, where they even out the
// CTAs' totals instead of adding to the longest.
__device__ __forceinline__ int g2_last_group_at(const int32_t* start, int32_t ngroups, int32_t t) {
  int lo = 0, hi = ngroups - 1;  // last selected group whose first tile <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ G2Tile g2_tile(int32_t t, const int32_t* tile_start, const int32_t* part_start,
                                          const int32_t* group_id, int32_t ngroups, int32_t n_full,
                                          const Gemm2Args& a, int32_t nb) {
  G2Tile ti;
  if (t < n_full) {
    const int i = g2_last_group_at(tile_start, ngroups, t);
    const int32_t local = t - tile_start[i];
    const int32_t mt = local / nb, ft = local - mt * nb;
    ti.g = group_id[i];
    ti.row0 = a.offsets[ti.g] + mt * g2::kN;
    ti.rows = g2::kN;
    ti.n0 = ft * g2::kM;
  } else {
    const int i = g2_last_group_at(part_start, ngroups, t - n_full);
    ti.g = group_id[i];
    const int32_t c = a.counts[ti.g], mt = c / g2::kN;
    ti.row0 = a.offsets[ti.g] + mt * g2::kN;
    ti.rows = c - mt * g2::kN;
    ti.n0 = (t - n_full - part_start[i]) * g2::kM;
  }
  return ti;
}

// Bounded wait that also gives up when another role has aborted.  Between
// polls the thread is suspended (try_wait with a time hint) rather than
// spinning: polling warps take shared-memory bandwidth from the MMA's operand
// reads.
__device__ __forceinline__ bool g2_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      if (err) atomicOr(err, kFlagTimeout);
      return false;
    }
  }
}

// Warps 1 and 2 meet at named barrier 2; returns the OR of `abort` over both
// (only warp 2 ever passes true).
__device__ __forceinline__ bool g2_handoff(bool abort) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 2, 64, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)abort)
      : "memory");
  return r != 0;
}

}  // namespace

__global__ void __launch_bounds__(g2::kThreads, 1)
    nvfp4_gemm2_kernel(const __grid_constant__ CUtensorMap tmX, const Gemm2Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + g2::bars);
  uint64_t* w_full = bars;                          // [kWStages] producer expect_tx
  uint64_t* w_empty = w_full + g2::kWStages;        // [kWStages] one arrival per unpack warp
  uint64_t* b_full = w_empty + g2::kWStages;        // [kBStages] producer expect_tx
  uint64_t* b_empty = b_full + g2::kBStages;        // [kBStages] MMA commit
  uint64_t* a_full = b_empty + g2::kBStages;        // [kAStages] one arrival per unpack warp
  uint64_t* a_empty = a_full + g2::kAStages;        // [kAStages] MMA commit
  uint64_t* tmem_full = a_empty + g2::kAStages;     // [2] MMA commit
  uint64_t* tmem_empty = tmem_full + 2;             // [2] one arrival per epilogue warp
  uint64_t* drain = tmem_empty + 2;                 // [1] final MMA commit
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + g2::misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + g2::misc + 8);
  int32_t* ngroups_sm = reinterpret_cast<int32_t*>(sm + g2::misc + 16);
  int32_t* total_sm = reinterpret_cast<int32_t*>(sm + g2::misc + 20);
  int32_t* tile_start = reinterpret_cast<int32_t*>(sm + g2::tile_start);
  int32_t* group_id = reinterpret_cast<int32_t*>(sm + g2::group_id);
  int32_t* part_start = reinterpret_cast<int32_t*>(sm + g2::part_start);
  uint32_t* lut = reinterpret_cast<uint32_t*>(sm + g2::scale_lut);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- set-up
  for (int i = tid; i < 256; i += g2::kThreads) lut[i] = scale_bf16_2p118((uint32_t)i) * 0x10001u;
  if (tid == 0) {
    for (int s = 0; s < g2::kWStages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], g2::kUnpackWarps);
    }
    for (int s = 0; s < g2::kBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < g2::kAStages; ++s) {
      mbar_init(&a_full[s], g2::kUnpackWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmX);
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }

  // Inputs (counts, packed activations) come from the previous kernel.
  pdl_wait();

  const int32_t nb = (a.N + g2::kM - 1) / g2::kM;
  if (warp == 3) {  // tile lists: selected groups in order, full token tiles, then the partial ones
    int32_t run = 0, prun = 0, ng = 0;
    for (int base = 0; base < a.G; base += 32) {
      const int g = base + lane;
      int32_t tiles = 0, ptiles = 0;
      bool sel = false;
      if (g < a.G) {
        const int32_t c = a.counts[g];
        sel = c > 0 && c > a.min_rows;
        if (sel) {
          tiles = (c / g2::kN) * nb;
          ptiles = (c % g2::kN) ? nb : 0;
        }
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, sel);
      int32_t incl = tiles, pincl = ptiles;
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
        const int32_t pv = __shfl_up_sync(0xffffffffu, pincl, d);
        if (lane >= d) {
          incl += v;
          pincl += pv;
        }
      }
      if (sel) {
        const int slot = ng + __popc(bal & ((1u << lane) - 1u));
        tile_start[slot] = run + incl - tiles;
        part_start[slot] = prun + pincl - ptiles;
        group_id[slot] = g;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      prun += __shfl_sync(0xffffffffu, pincl, 31);
      ng += __popc(bal);
    }
    if (lane == 0) {
      *ngroups_sm = ng;
      *total_sm = run + prun;
      *(total_sm + 1) = run;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t ngroups = *ngroups_sm, total_tiles = *total_sm, n_full = *(total_sm + 1);
  pdl_launch_dependents();

  const int32_t KB = a.K / g2::kK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One thread: the waits of a full warp on already-completed barriers
    // cost more than the copies they gate.
    if (lane == 0) {
      int ws = 0, bs = 0;
      uint32_t wph = 0, bph = 0;
      uint32_t w_out = 0, b_out = 0;  // stages whose last fill may still be landing
      uint32_t w_iss[g2::kWStages] = {}, b_iss[g2::kBStages] = {};
      bool ok = true;
      for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const G2Tile ti = g2_tile(t, tile_start, part_start, group_id, ngroups, n_full, a, nb);
        const uint8_t* wsrc = a.blocks + ((size_t)ti.g * nb + ti.n0 / g2::kM) * KB * (size_t)g2::kWBytes;
        for (int32_t kb = 0; kb < KB; ++kb) {
          if (!g2_wait(&w_empty[ws], wph ^ 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&w_full[ws], g2::kWBytes);
          bulk_g2s(sm + g2::w + ws * g2::kWBytes, wsrc + (size_t)kb * g2::kWBytes, g2::kWBytes, &w_full[ws]);
          w_out |= 1u << ws;
          w_iss[ws] = wph;
          if (++ws == g2::kWStages) {
            ws = 0;
            wph ^= 1u;
          }
          if (!g2_wait(&b_empty[bs], bph ^ 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], g2::kBBytes);
          tma_load_2d(sm + g2::b + bs * g2::kBBytes, &tmX, kb * g2::kK, ti.row0, &b_full[bs]);
          b_out |= 1u << bs;
          b_iss[bs] = bph;
          if (++bs == g2::kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      if (!ok) {
        // Unwinding: let every copy issued here land before the CTA exits
        // (bounded: 1 ms per stage).
        for (int s = 0; s < g2::kWStages; ++s) {
          if (!(w_out & (1u << s))) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&w_full[s], w_iss[s]) && globaltimer_ns() - t0 < 1000000ull) {
          }
        }
        for (int s = 0; s < g2::kBStages; ++s) {
          if (!(b_out & (1u << s))) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&b_full[s], b_iss[s]) && globaltimer_ns() - t0 < 1000000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // A shared-memory load by the thread that issued tcgen05.mma waits until
    // those MMAs have read their shared-memory operands, draining the tensor
    // core's shallow queue; so this warp reads no shared memory per k-block.
    // Warp 2 waits on the stage barriers and hands each k-block over through
    // named barrier 2 (no memory access), with an abort bit riding along.
    int bs = 0, as = 0, it = 0;
    bool done = false;
    // descriptor of stage 0, k 0; the start-address field (address >> 4, low
    // 14 bits) of the others is this plus the byte offset >> 4, no carry for
    // offsets inside shared memory
    const uint64_t bdesc0 = smem_desc_k128(smem_u32(sm + g2::b));
    for (int32_t t = blockIdx.x; t < total_tiles && !done; t += gridDim.x, ++it) {
      const G2Tile ti = g2_tile(t, tile_start, part_start, group_id, ngroups, n_full, a, nb);  // once per tile
      const uint32_t acc = it & 1;
      const uint32_t ncols = (uint32_t)((ti.rows + 15) & ~15);
      const uint32_t idesc = idesc_bf16(g2::kM, ncols);
      const uint32_t d_tmem = tmem_base + acc * g2::kAccCols;
      for (int32_t kb = 0; kb < KB; ++kb) {
        if (g2_handoff(false)) {
          done = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)(bs * g2::kBBytes) >> 4);
          const uint32_t a_tmem = tmem_base + g2::kACol0 + as * g2::kAStageCols;
          tc_mma_bf16_ta(d_tmem, a_tmem, bd, idesc, kb != 0);
#pragma unroll
          for (int kk = 1; kk < g2::kK / 16; ++kk) tc_mma_bf16_ta(d_tmem, a_tmem + kk * 8, bd + 2 * kk, idesc, 1);
          tc_commit(&b_empty[bs]);
          tc_commit(&a_empty[as]);
        }
        if (++bs == g2::kBStages) bs = 0;
        if (++as == g2::kAStages) as = 0;
      }
      if (done) break;
      if (lane == 0) tc_commit(&tmem_full[acc]);
      __syncwarp();
    }
    // all MMAs issued here have completed once `drain` flips
    if (lane == 0) {
      tc_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ readiness
    // For each k-block of the MMA issuer's sequence: the accumulator is free
    // (first k-block of a tile), the activation tile and the unpacked weights
    // have landed; then the hand-off.  Same trip count as the issuer.
    int bs = 0, as = 0, it = 0;
    uint32_t bph = 0, aph = 0;
    bool done = false;
    for (int32_t t = blockIdx.x; t < total_tiles && !done; t += gridDim.x, ++it) {
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      for (int32_t kb = 0; kb < KB; ++kb) {
        bool fail = false;
        if (lane == 0) {
          if (kb == 0) fail = !g2_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, a.err);
          fail = fail || !g2_wait(&b_full[bs], bph, abort_flag, a.err) ||
                 !g2_wait(&a_full[as], aph, abort_flag, a.err);
        }
        __syncwarp();
        if (g2_handoff(fail)) {
          done = true;
          break;
        }
        if (++bs == g2::kBStages) {
          bs = 0;
          bph ^= 1u;
        }
        if (++as == g2::kAStages) {
          as = 0;
          aph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 4 + g2::kUnpackGroups * g2::kUnpackWarps) {
    // ------------------------------------------------------------ unpack
    // k-block L (counted over this CTA's tiles) uses weight stage L % 8
    // (phase (L / 8) & 1) and A stage L % kAStages (phase (L / kAStages) & 1);
    // group L % 2 unpacks it.
    const int q = warp & 3;                        // TMEM lanes 32q .. 32q+31
    const int hf = ((warp - 4) >> 2) & 1;          // k 32hf .. 32hf+31 of the block
    const int grp = (warp - 4) >> 3;
    const int row = 32 * q + lane;
    const uint32_t col_off = ((uint32_t)(32 * q) << 16) + g2::kACol0 + hf * 16;
    const int cswap = (row >> 2) & 1;
    bool ok = true;
    int32_t L = 0;
    for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      for (int32_t kb = 0; kb < KB; ++kb, ++L) {
        if ((L & 1) != grp) continue;
        static_assert(g2::kWStages == 8, "stage arithmetic below");
        const int sw = L & 7, s = L % g2::kAStages;
        const uint32_t wph = (uint32_t)(L >> 3) & 1u, ph = (uint32_t)(L / g2::kAStages) & 1u;
        if (!g2_wait(&w_full[sw], wph, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint8_t* wb = sm + g2::w + sw * g2::kWBytes;
        const uint4 c = *reinterpret_cast<const uint4*>(wb + row * 32 + ((hf ^ cswap) << 4));
        const uint32_t sc = *reinterpret_cast<const uint16_t*>(wb + 4096 + row * 4 + 2 * hf);
        const uint32_t s0 = lut[sc & 0xFFu], s1 = lut[sc >> 8];
        __syncwarp();
        if (lane == 0) mbar_arrive(&w_empty[sw]);  // release: the reads above are done
        uint32_t r[16];
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t p0, p1, p2, p3;
          unpack_word(words[j], p0, p1, p2, p3);
          const uint32_t sv = j < 2 ? s0 : s1;
          r[4 * j + 0] = mul_bf16x2(p0, sv);
          r[4 * j + 1] = mul_bf16x2(p1, sv);
          r[4 * j + 2] = mul_bf16x2(p2, sv);
          r[4 * j + 3] = mul_bf16x2(p3, sv);
        }
        if (!g2_wait(&a_empty[s], ph ^ 1u, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tmem_base + col_off + s * g2::kAStageCols, r);
        // signal the stage as soon as the store has landed: the A stages are
        // the tightest buffer between the unpack and the MMA
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
      }
    }
  } else if (warp >= 4 + g2::kUnpackGroups * g2::kUnpackWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31: feature rows
    const int row = 32 * q + lane;
    int it = 0;
    for (int32_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const G2Tile ti = g2_tile(t, tile_start, part_start, group_id, ngroups, n_full, a, nb);
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      if (!g2_wait(&tmem_full[acc], acc_phase, abort_flag, a.err)) break;
      tc_fence_after();
      const int32_t f = ti.n0 + row;
      const bool live = f < a.N;
      const float alpha = a.global[ti.g] * 256.0f;  // the unpacked weights carry 2^-8
      const int32_t ncols = (ti.rows + 15) & ~15;
      if (a.epilogue == 2) {
        // lanes 0-15 hold the gate rows of features n0/2 + 16q + lane, lanes
        // 16-31 the up rows.  Per pair of token columns (i, i+1) one shuffle
        // hands the low half the up value of column i and the high half the
        // gate value of column i+1, so every lane finishes one output.
        const bool lo = lane < 16;
        const float ah = lo ? a.global2[ti.g] * 256.0f : alpha;
        const int32_t NO = a.N / 2;
        const int32_t fo = ti.n0 / 2 + 16 * q + (lane & 15);
        for (int32_t c0 = 0; c0 < ncols; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + acc * g2::kAccCols + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float h0 = ah * __uint_as_float(r[i]), h1 = ah * __uint_as_float(r[i + 1]);
            const float got = __shfl_xor_sync(0xffffffffu, lo ? h1 : h0, 16);
            const float gv = lo ? h0 : got, uv = lo ? got : h1;
            const int32_t tok = c0 + i + (lo ? 0 : 1);
            // silu(g) = g / (1 + e^-g), fast exponential and divide: the
            // result is rounded to bf16, far coarser than their error
            const float av = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            if (tok < ti.rows && live)
              reinterpret_cast<uint16_t*>(a.out)[(size_t)(ti.row0 + tok) * NO + fo] = f2bf_rn(av);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[acc]);
        continue;
      }
      for (int32_t c0 = 0; c0 < ncols; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + acc * g2::kAccCols + c0, r);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int32_t tok = c0 + i;
            if (tok < ti.rows) {
              const size_t o = (size_t)(ti.row0 + tok) * a.N + f;
              const float h = alpha * __uint_as_float(r[i]);
              if (a.epilogue == 1) {
                const float rl = fmaxf(h, 0.f);
                reinterpret_cast<uint16_t*>(a.out)[o] = f2bf_rn(rl * rl);
              } else {
                reinterpret_cast<float*>(a.out)[o] = h;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[acc]);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t launch_gemm2(const CUtensorMap& tmX, const Gemm2Args& a, int num_sms, cudaStream_t s, bool pdl) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = raise_smem_limit(nvfp4_gemm2_kernel, (int)g2::alloc, configured);
  if (e != cudaSuccess) return e;
  return launch_ex(nvfp4_gemm2_kernel, dim3(num_sms > 0 ? num_sms : 1), dim3(g2::kThreads), g2::alloc, s, pdl, tmX,
                   a);
}

}  // namespace moe
