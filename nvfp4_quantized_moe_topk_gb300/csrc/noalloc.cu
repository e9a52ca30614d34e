// noalloc.cu -- a forward of the layer that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code running inside a host program
// that owns every byte of device memory through its own pool (an inference
// server or plugin host that must account for all allocations), callers with
// a fixed memory budget decided at load time, and callers that must not
// trigger the implicit device synchronisation cudaMalloc may cause.  For them
// this entry point takes the weights and activations as given and keeps every
// intermediate (routing arrays, relu^2 or silu*up rows, down rows, error flag) in one
// file-scope __device__ array of fixed size, which every GPU that loads the
// library holds until the process exits.
//
// Set-up: the first call on a device looks up that device's address of the
// array with cudaGetSymbolAddress (with the device current) and caches it;
// make that first call before any stream capture.  All calls on a device
// share its one array and it keeps the last call's contents: calls whose work
// overlaps on the GPU (for example on two streams) race on it, so the caller
// must order them.
// The kernels are the same routing / weight-streaming GEMV / combine kernels
// the handle-based forward uses on its small-batch path.
#include <mutex>

#include "../../include/moe_nvfp4.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
using moe::kMaxDevices;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

extern "C" moe_status moe_nvfp4_forward_noalloc(const moe_nvfp4_config* config, const moe_nvfp4_weights* w,
                                                const uint16_t* x, const int32_t* topk_ids,
                                                const float* topk_weights, uint16_t* dst, int32_t n_tokens,
                                                moe_stream_t stream) {
  if (!config || !w || n_tokens < 0) return MOE_ERR_INVALID_ARG;
  const int H = config->hidden, I = config->inter, E = config->n_experts, k = config->top_k;
  if (H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 || I % 64 || E > 1024 || k > 32 || H > 4096 || I > 4096) return MOE_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_weights || !dst || !w->up_codes || !w->up_scales || !w->down_codes ||
      !w->down_scales || !w->up_global || !w->down_global)
    return MOE_ERR_INVALID_ARG;
  if (config->activation != MOE_ACT_RELU2 && config->activation != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  const bool gated = config->activation == MOE_ACT_SWIGLU;
  if (gated && (!w->gate_codes || !w->gate_scales || !w->gate_global)) return MOE_ERR_INVALID_ARG;
  // The kernels read codes, x and dst 16 bytes at a time, scales 2 bytes at a
  // time and globals, ids and weights as 4-byte words: a pointer off those
  // boundaries is an argument error, not a misaligned access on the GPU.
  auto misaligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (misaligned(x, 16) || misaligned(dst, 16) || misaligned(w->up_codes, 16) || misaligned(w->down_codes, 16) ||
      misaligned(w->up_scales, 2) || misaligned(w->down_scales, 2) || misaligned(w->up_global, 4) ||
      misaligned(w->down_global, 4) || misaligned(topk_ids, 4) || misaligned(topk_weights, 4))
    return MOE_ERR_INVALID_ARG;
  if (gated && (misaligned(w->gate_codes, 16) || misaligned(w->gate_scales, 2) || misaligned(w->gate_global, 4)))
    return MOE_ERR_INVALID_ARG;

  // Carve the fixed array: routing arrays, error flag, slice histograms, relu^2 rows, down rows.
  const size_t R = (size_t)n_tokens * k;
  size_t off = 0;
  const size_t o_counts = off;
  off = round_up(off + 4 * (size_t)E, 256);
  const size_t o_offsets = off;
  off = round_up(off + 4 * ((size_t)E + 1), 256);
  const size_t o_perm = off;
  off = round_up(off + 4 * R, 256);
  const size_t o_inv = off;
  off = round_up(off + 4 * R, 256);
  const size_t o_err = off;
  off = round_up(off + 4, 256);
  const size_t o_blk = off;
  off = round_up(off + 4 * (moe::routing_scratch_ints((int64_t)R, E) + 1), 256);
  const size_t o_ap = off;
  off = round_up(off + 2 * R * (size_t)I, 256);
  const size_t o_yp = off;
  off = round_up(off + 4 * R * (size_t)H, 256);
  if (off > kNoAllocScratchBytes) return MOE_ERR_CAPACITY;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    base = static_cast<unsigned char*>(g_noalloc_addr[dev]);
  }
  int32_t* counts = reinterpret_cast<int32_t*>(base + o_counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + o_offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + o_perm);
  int32_t* inv = reinterpret_cast<int32_t*>(base + o_inv);
  int32_t* err = reinterpret_cast<int32_t*>(base + o_err);
  int32_t* blk_hist = reinterpret_cast<int32_t*>(base + o_blk);
  uint16_t* Ap = reinterpret_cast<uint16_t*>(base + o_ap);
  float* Yp = reinterpret_cast<float*>(base + o_yp);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The error flag is the only piece of the array that must start at zero
  // (the kernels overwrite every other word they read).
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_routing(topk_ids, (int32_t)R, E, counts, offsets, perm, inv, err, s, blk_hist) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe::GemvArgs g{};
  g.counts = counts;
  g.offsets = offsets;
  g.perm_pair = perm;
  g.E = E;
  g.k = k;
  g.max_rows = 0;  // every expert through the weight-streaming kernel
  g.codes = w->up_codes;
  g.scales = w->up_scales;
  g.global = w->up_global;
  g.in = x;
  g.out = Ap;
  g.N = I;
  g.K = H;
  g.token_indexed = 1;
  g.relu2_bf16_out = 1;
  if (gated) {
    g.gate_codes = w->gate_codes;
    g.gate_scales = w->gate_scales;
    g.gate_global = w->gate_global;
  }
  if (moe::launch_gemv(g, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  g.gate_codes = nullptr;
  g.gate_scales = nullptr;
  g.gate_global = nullptr;
  g.codes = w->down_codes;
  g.scales = w->down_scales;
  g.global = w->down_global;
  g.in = Ap;
  g.out = Yp;
  g.N = H;
  g.K = I;
  g.token_indexed = 0;
  g.relu2_bf16_out = 0;
  if (moe::launch_gemv(g, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_weighted_row_sum(dst, Yp, inv, topk_weights, n_tokens, k, H, (int32_t)R, s, true) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
