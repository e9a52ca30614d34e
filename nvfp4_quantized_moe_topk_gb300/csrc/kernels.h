// kernels.h -- internal launchers of libmoe_nvfp4 (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace moe {

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device.  The per-device flags are atomics because launches may come from
// several host threads; two threads setting the attribute at once is harmless.
constexpr int kMaxDevices = 64;
template <typename Kernel>
inline cudaError_t raise_smem_limit(Kernel* kernel, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
  return e;
}

// ---------------------------------------------------------------- routing
// Pairs per routing slice (one CTA each); batches of more than one slice need
// routing_scratch_ints(R, E) ints of device scratch for the slice histograms.
constexpr int kRoutingSlice = 4096;
size_t routing_smem_bytes(int E);
size_t routing_scratch_ints(int64_t R, int E);
cudaError_t launch_routing(const int32_t* ids, int32_t R, int32_t E, int32_t* counts, int32_t* offsets,
                           int32_t* perm_pair, int32_t* inv, int32_t* err, cudaStream_t s, int32_t* blk_hist);

// ------------------------------------------------------------------ router
// ids/w [n][k] from fp32 logits [n][E] (+ bias [E] or nullptr); counts [E]
// (or nullptr) is zeroed and receives the pick histogram.  k <= 32.
cudaError_t launch_router(const float* logits, const float* bias, int32_t n, int32_t E, int32_t k, int32_t* ids,
                          float* w, int32_t* counts, cudaStream_t s);

// ------------------------------------------------------------ gather / combine
// Xp[inv[t*k + j]][:] = x[t][:] for every pair with 0 <= inv < R (n tokens).
cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int32_t n, int32_t k, int32_t H, int32_t R,
                          uint16_t* Xp, cudaStream_t s, bool pdl);
// dst[i][c] = bf16(dst[i][c] + sum_j w[i][j] * src[rows[i][j]][c]), fixed j order.
cudaError_t launch_weighted_row_sum(uint16_t* dst, const float* src, const int32_t* rows, const float* w,
                                    int32_t n, int32_t k, int32_t cols, int32_t src_rows, cudaStream_t s,
                                    bool pdl);

// ------------------------------------------------------------ NVFP4 GEMV
// Weight-streaming matrix-vector path for experts with few rows.
struct GemvArgs {
  const uint8_t* codes;    // [E][N][K/2]
  const uint8_t* scales;   // [E][N][K/16]
  const float* global;     // [E]
  const int32_t* counts;   // [E]
  const int32_t* offsets;  // [E+1]
  const int32_t* perm_pair;  // [R] (token-indexed input only)
  const uint16_t* in;      // bf16: x [n][K] (token-indexed) or Ap [R][K] (row-indexed)
  void* out;               // bf16 Ap [R][N] (relu^2) or fp32 Yp [R][N]
  int32_t E, N, K, k;
  int32_t max_rows;        // experts with 0 < count <= max_rows take this path (<= 0: every expert)
  int32_t token_indexed;   // 1: input row of packed row r is in[perm_pair[r] / k]
  int32_t relu2_bf16_out;  // 1: out = bf16(max(g*acc,0)^2); 0: out = fp32 g*acc
  // non-null: gated up projection, out = bf16(silu(gg*gate_acc) * g*acc)
  const uint8_t* gate_codes;   // [E][N][K/2]
  const uint8_t* gate_scales;  // [E][N][K/16]
  const float* gate_global;    // [E]
};
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl);

// ------------------------------------------------------- tcgen05 grouped GEMM
struct GemmArgs {
  const uint8_t* scales;   // [G][N][K/16] (G groups of N weight rows)
  const float* global;     // [G] per-group alpha, or nullptr to use alpha0
  float alpha0;
  const int32_t* counts;   // [G] rows per group, or nullptr: single group of M rows
  const int32_t* offsets;  // [G+1]
  int32_t M;               // single-group row count (counts == nullptr)
  int32_t G, N, K;
  int32_t min_rows;        // groups with count > min_rows take this path (grouped mode)
  void* out;               // [rows][N]: fp32 (epilogue 0) or bf16 relu^2 (epilogue 1)
  int32_t epilogue;
  int32_t* err;            // device error flag (may be nullptr)
};
// tmA: bf16 activations [rows][K], box 64 x 128, 128-byte swizzle.
// tmB: weight codes [G*N][K/2] bytes, box 32 x 256, no swizzle.
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int num_sms,
                        cudaStream_t s, bool pdl);

// ------------------------------------------- grouped GEMM, A operand in TMEM
// Packed weight blocks [G][ceil(N/128)][K/64] of 4608 bytes (gemm2.cu).
constexpr uint32_t kGemmBlockBytes = 128 * 32 + 128 * 4;
constexpr int kGemmTileRows = 224;  // packed rows (tokens) per grouped-GEMM tile
cudaError_t launch_repack_gemm(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                               uint8_t* out, cudaStream_t s);
size_t gemm_blocks_bytes(int32_t G, int32_t N, int32_t K);
struct Gemm2Args {
  const uint8_t* blocks;   // packed weight blocks of the G groups
  const float* global;     // [G] per-group alpha
  const int32_t* counts;   // [G] rows per group
  const int32_t* offsets;  // [G+1]
  int32_t G, N, K;
  int32_t min_rows;        // groups with count > min_rows take this path
  void* out;               // [rows][N]: fp32 (epilogue 0) or bf16 relu^2 (epilogue 1);
                           // [rows][N/2] bf16 silu(gate) * up (epilogue 2)
  int32_t epilogue;
  const float* global2;    // [G] gate alpha (epilogue 2: rows in groups of 16 gate then 16 up)
  int32_t* err;
};
// tmX: bf16 activations [rows][K], box 64 x kGemmTileRows, 128-byte swizzle.
cudaError_t launch_gemm2(const CUtensorMap& tmX, const Gemm2Args& a, int num_sms, cudaStream_t s, bool pdl);
cudaError_t make_tmap_act_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows);

// ------------------------------------------------------- decode (small batch)
// Fragment-tile weight layout and the single-launch small-batch layer (decode.cu).
constexpr int kTileBytes = 576;        // 16 rows x 64 k: 512 code bytes + 64 scale bytes
constexpr int kDecMaxWarps = 16;       // warps per CTA
constexpr int kDecMaxSlots = 8;        // weight-ring slots per warp (at most)
constexpr int kDecCK = 4;              // k-tiles (of 64) per chunk
constexpr int kDecSlotBytes = 2 * kDecCK * kTileBytes;  // weights of a chunk: 2 row tiles x kDecCK k-tiles
constexpr int kDecPassTok = 8;         // tokens per pass over a tile (one n8 MMA block)
constexpr int kDecL2Ahead = 8;         // chunks past the ring requested into L2 at start
constexpr long long kDecEarlyL2Bytes = 48ll << 20;  // picked experts' up weights prefetched during routing, at most
constexpr int kDecLateCombine = 8;     // larger batches combine after a second grid barrier
// Partial sums of split items, per CTA: (warp, first/last segment) x 32 lanes x
// 2 float4.  The kernel that can stage keeps them in global memory (an
// L1-resident 32 KB per SM) so that the shared memory goes to the ring and
// the stage; the one-token kernel keeps them in shared memory.
constexpr int kDecPartialPerCta = 2 * kDecMaxWarps * 32 * 2;  // float4
constexpr int kDecMaxSpan = 16;        // experts whose activation rows one CTA stages per phase, at most
constexpr int kDecStageMax = 96 * 1024;  // bytes of staged activation rows per CTA, at most
constexpr int kDecMaxPairs = 1024;     // batches with at most this many pairs
constexpr int kDecMaxTokens = 64;      // and tokens run as one launch

// Shared-memory plan of the decode kernel (byte offsets; the host computes it).
struct DecLayout {
  uint32_t scale_lut, scale_lut16, ids, perm, inv, counts, offsets, act, misc, bars, partial, pcount, desc, sbase,
      rowexp, ring, total;
  uint32_t warps;
};

inline DecLayout dec_layout(int32_t E, int32_t R, uint32_t budget, bool smem_partial) {
  DecLayout L{};
  uint32_t o = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    o = (o + align - 1) / align * align;
    const uint32_t at = o;
    o += bytes;
    return at;
  };
  L.scale_lut = take(256 * 4, 128);
  L.scale_lut16 = take(256 * 4, 128);
  L.ids = take(4 * (uint32_t)R, 16);
  L.perm = take(4 * (uint32_t)R, 16);
  L.inv = take(4 * (uint32_t)R, 16);
  L.counts = take(4 * (uint32_t)E, 16);
  L.offsets = take(4 * ((uint32_t)E + 1), 16);
  L.act = take(4 * (uint32_t)E, 16);
  L.misc = take(64, 16);
  L.bars = take(8 * (kDecMaxSlots * kDecMaxWarps + 1), 16);  // ring slots, then the stage barrier
  L.partial = smem_partial ? take(kDecPartialPerCta * 16, 128) : 0;
  L.pcount = take(kDecMaxWarps * 4, 16);
  L.desc = take(kDecMaxWarps * kDecMaxSlots * 48, 16);  // per-slot chunk descriptors
  L.sbase = take(4 * 2 * (kDecMaxSpan + 1), 16);        // per phase: first stage row of each staged expert
  L.rowexp = take(4 * kDecPassTok * kDecMaxSpan, 16);   // power-of-two exponent of each staged row
  const uint32_t ring_at = (o + 127) / 128 * 128;
  uint32_t warps = budget > ring_at ? (budget - ring_at) / (2 * kDecSlotBytes) : 0;
  if (warps > (uint32_t)kDecMaxWarps) warps = kDecMaxWarps;
  L.warps = warps;
  L.ring = ring_at;
  L.total = budget;
  return L;
}

struct DecodeArgs {
  const uint8_t* up_tiles;    // [E][I/16][H/64][576]; gated: [E][2I/16][H/64][576], gate and up tiles alternating
  const uint8_t* dn_tiles;    // [E][H/16][I/64][576]
  const uint8_t* up_tiles16;  // the same tiles with codes in byte order for the f16 path (launch_repack_frag16)
  const uint8_t* dn_tiles16;
  const float* up_g;
  const float* dn_g;
  const float* gate_g;        // gated only
  int32_t gated;              // 1: a = bf16(silu(gate) * up), else bf16(relu(up)^2)
  const uint16_t* x;          // [n][H] bf16
  const int32_t* ids;         // [n][k]
  const float* tw;            // [n][k]
  uint16_t* dst;              // [n][H] bf16
  uint16_t* dst_out;          // [n][H] bf16: where the in-kernel combine writes (dst, or a host-mapped copy of it)
  uint16_t* Ap;               // [R][I] bf16 (workspace)
  float* Yp;                  // [R][H] fp32 (workspace)
  int32_t* g_counts;          // routing results kept for the debug entry point
  int32_t* g_offsets;
  int32_t* g_perm;
  int32_t* g_inv;
  int32_t* col_done;          // [H/16] combine counters, zero between launches
  float4* partial;            // [gridDim.x][kDecPartialPerCta] split-item partial sums (scratch)
  int32_t* grid_bar;          // 8-byte aligned: one 64-bit arrival count (multiple of the grid between launches)
  int32_t* err;
  int32_t n, H, I, E, k;
  // ext = 1: routing comes from g_counts / g_offsets / g_perm (written by the
  // routing kernel), only experts with 0 < count <= max_rows are processed,
  // and the combine is left to the WeightedRowSum kernel.
  int32_t ext, max_rows;
  DecLayout L;
};

cudaError_t launch_repack_frag(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                               uint8_t* out, cudaStream_t s);
cudaError_t launch_repack_frag16(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                                 uint8_t* out, cudaStream_t s);
// Shared-memory plan for E experts and R pairs (227 KB budget), for the
// kernel launch_decode picks for these arguments.
DecLayout decode_layout(int32_t E, int32_t R, bool can_stage);
// The streaming kernel that can stage activation rows (several tokens, or
// external routing); one-token batches take the per-chunk kernel alone.
inline bool decode_can_stage(int32_t n, int32_t ext) { return n > 1 || ext; }
cudaError_t launch_decode(const DecodeArgs& args, int num_sms, cudaStream_t s);

// Host helpers for tensor maps (driver entry point resolved at run time).
cudaError_t make_tmap_act(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K);
cudaError_t make_tmap_codes(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K);

// Launch with the programmatic-stream-serialization attribute when pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
