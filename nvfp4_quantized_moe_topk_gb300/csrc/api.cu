// api.cu -- the C ABI of libmoe_nvfp4 (declared in include/moe_nvfp4.h).
//
// Host side of the layer: argument validation (every failure returns a status
// before anything is enqueued), ownership of the weights and of one workspace
// sized for max_tokens at create time (gllm pull request #91, "Results":
// per-op cudaMalloc/cudaFree and a synchronisation on every op were what
// remained of the host cost, so forward allocates nothing and never waits),
// tensor-map construction, and the launch sequence of one forward:
//
//   n <= single_max_tokens (64) and n*k <= 1024: one cooperative launch of the streaming kernel
//   (routing, up, relu^2, down and the combine in one kernel)
//   otherwise: routing -> gather -> streaming kernel for experts with at most
//   T rows (both projections) -> tcgen05 grouped GEMM up -> grouped GEMM down
//   -> WeightedRowSum
//
// Gated experts (silu(gate) * up): create interleaves the gate and up
// matrices in groups of 16 rows (16 gate rows, then the 16 up rows of the
// same features) into one 2I-row matrix and repacks that for both kernels, so
// a streaming-kernel work item is a (gate, up) tile pair and a grouped-GEMM
// weight block holds 64 features' gate and up rows.
//
// chained with programmatic dependent launch so each kernel's prologue
// overlaps its predecessor's tail.  The GEMM kernels are enqueued only when
// some expert can exceed the threshold T (n > T); which experts take which
// path is decided on the device from the routing counts.  When T is set so
// large that no expert can exceed it and the batch is too large for one
// launch, the GEMV kernels serve every expert.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe_nvfp4.h"
#include "kernels.h"

namespace {

using namespace moe;

enum KernelId {
  kKRouting = 0, kKGather, kKGemvUp, kKGemmUp, kKGemvDown, kKGemmDown, kKCombine, kKDecode, kKSmall, kKCount
};
const char* const kKernelNames[kKCount] = {"routing",   "gather",    "gemv_up", "gemm_up",      "gemv_down",
                                           "gemm_down", "combine",   "decode",  "small_experts"};
// The same names as NVTX ranges (what a profiler shows around each launch).
const char* const kRangeNames[kKCount] = {"moe_nvfp4/routing",   "moe_nvfp4/gather",  "moe_nvfp4/gemv_up",
                                          "moe_nvfp4/gemm_up",   "moe_nvfp4/gemv_down", "moe_nvfp4/gemm_down",
                                          "moe_nvfp4/combine",   "moe_nvfp4/decode",  "moe_nvfp4/small_experts"};

struct TimingSlot {
  cudaEvent_t beg = nullptr, end = nullptr;
  int kernel = -1;
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr size_t kSmallStage = 64 * 1024;  // bytes; below this a host call packs its inputs
size_t round16(size_t v) { return (v + 15) & ~size_t(15); }

}  // namespace

struct moe_nvfp4 {
  moe_nvfp4_config cfg{};
  int device = 0;
  int num_sms = 0;
  int threshold = 8;
  int single_max_tokens = kDecMaxTokens;
  // library-owned weights
  uint8_t *up_codes = nullptr, *up_scales = nullptr, *dn_codes = nullptr, *dn_scales = nullptr;
  float *up_g = nullptr, *dn_g = nullptr;
  bool gated = false;
  uint8_t *gate_codes = nullptr, *gate_scales = nullptr;
  float* gate_g = nullptr;
  // the same weights in fragment-tile order for the single-launch small-batch path
  uint8_t *up_tiles = nullptr, *dn_tiles = nullptr;
  // and with whole code bytes in fragment order for its f16 path (batches of several tokens)
  uint8_t *up_tiles16 = nullptr, *dn_tiles16 = nullptr;
  // and in packed 128-row blocks for the grouped GEMM
  uint8_t *up_blocks = nullptr, *dn_blocks = nullptr;
  int32_t *col_done = nullptr, *grid_bar = nullptr;
  float4* dec_partial = nullptr;  // streaming kernel: split-item partial sums, per CTA
  // workspace (max_tokens)
  int32_t *counts = nullptr, *offsets = nullptr, *perm_pair = nullptr, *inv = nullptr, *err = nullptr;
  int32_t* blk_hist = nullptr;  // per-slice expert histograms of the routing kernels
  // one-expert top-1 handles (shared expert): every token to expert 0 at weight 1
  int32_t* dense_ids = nullptr;
  float* dense_w = nullptr;
  uint16_t *Xp = nullptr, *Ap = nullptr;
  float* Yp = nullptr;
  // staging for forward_host
  uint16_t *x_stage = nullptr, *dst_stage = nullptr;
  int32_t* ids_stage = nullptr;
  float* w_stage = nullptr;
  // small host calls: the four inputs packed in one pinned host buffer and
  // moved by one copy each way (nullptr if the pinned allocation failed)
  uint8_t *small_dev = nullptr, *small_host = nullptr;
  uint8_t* small_host_dev = nullptr;  // small_host as the device sees it (mapped), or null
  // large host calls: dst's copy in runs on a side stream while the layer
  // computes; the combine waits for it (nullptr if creation failed)
  cudaStream_t side = nullptr;
  cudaEvent_t dst_in = nullptr;
  cudaEvent_t part_done[4] = {};  // combine chunks finished (their dst rows go back on the side stream)
  // tensor maps
  CUtensorMap tm_xp{}, tm_ap{};  // kGemmTileRows-row activation tiles of the grouped GEMM
  int32_t last_n = 0;
  // per-kernel timing
  bool timing = false;
  std::vector<TimingSlot> slots;
  size_t slot_next = 0;
  double total_ms[kKCount] = {};
  int64_t launches[kKCount] = {};
};

namespace {

void free_handle(moe_nvfp4* h) {
  if (!h) return;
  void* ptrs[] = {h->up_codes, h->up_scales, h->dn_codes, h->dn_scales, h->up_g,      h->dn_g,
                  h->counts,   h->offsets,   h->perm_pair, h->inv,      h->err,       h->Xp,
                  h->Ap,       h->Yp,        h->x_stage,   h->dst_stage, h->ids_stage, h->w_stage,
                  h->up_tiles, h->dn_tiles,  h->col_done,  h->grid_bar,  h->up_blocks, h->dn_blocks,
                  h->up_tiles16, h->dn_tiles16, h->dec_partial,
                  h->gate_codes, h->gate_scales, h->gate_g, h->blk_hist, h->dense_ids, h->dense_w};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->small_dev) cudaFree(h->small_dev);
  if (h->small_host) cudaFreeHost(h->small_host);
  if (h->dst_in) cudaEventDestroy(h->dst_in);
  for (cudaEvent_t ev : h->part_done)
    if (ev) cudaEventDestroy(ev);
  if (h->side) cudaStreamDestroy(h->side);
  for (auto& s : h->slots) {
    if (s.beg) cudaEventDestroy(s.beg);
    if (s.end) cudaEventDestroy(s.end);
  }
  delete h;
}

moe_status check_shape(int H, int I, int E, int k) {
  if (H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 || I % 64 || E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
  if (H > 4096 || I > 4096) return MOE_ERR_UNSUPPORTED;  // GEMV lane plan covers K <= 4096
  return MOE_OK;
}

int device_sms(int dev) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

bool is_sm103(int dev) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

// Brackets one kernel launch with an NVTX range (a no-op unless a profiler
// is attached) and, when timing is on, with timing events.
struct TimedLaunch {
  moe_nvfp4* h;
  cudaStream_t s;
  TimingSlot* slot = nullptr;
  TimedLaunch(moe_nvfp4* h_, cudaStream_t s_, int kernel) : h(h_), s(s_) {
    nvtxRangePushA(kRangeNames[kernel]);
    if (!h || !h->timing || h->slots.empty()) return;
    slot = &h->slots[h->slot_next];
    h->slot_next = (h->slot_next + 1) % h->slots.size();
    if (slot->kernel >= 0) {  // ring wrapped: fold the old measurement in first
      float ms = 0.f;
      if (cudaEventSynchronize(slot->end) == cudaSuccess && cudaEventElapsedTime(&ms, slot->beg, slot->end) == cudaSuccess) {
        h->total_ms[slot->kernel] += ms;
        h->launches[slot->kernel] += 1;
      }
    }
    slot->kernel = kernel;
    cudaEventRecord(slot->beg, s);
  }
  ~TimedLaunch() {
    if (slot) cudaEventRecord(slot->end, s);
    nvtxRangePop();
  }
};

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* moe_nvfp4_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CAPACITY: return "n_tokens exceeds max_tokens";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_ROUTING: return "expert id out of range (pair dropped)";
    case MOE_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    case MOE_ERR_NO_DEVICE: return "no sm_103 CUDA device";
  }
  return "unknown status";
}

moe_status moe_nvfp4_create(const moe_nvfp4_config* config, const moe_nvfp4_weights* w, moe_stream_t stream,
                            moe_nvfp4_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config || !w) return MOE_ERR_INVALID_ARG;
  if (!w->up_codes || !w->up_scales || !w->down_codes || !w->down_scales || !w->up_global || !w->down_global)
    return MOE_ERR_INVALID_ARG;
  const moe_nvfp4_config c = *config;
  if (c.activation != MOE_ACT_RELU2 && c.activation != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  const bool gated = c.activation == MOE_ACT_SWIGLU;
  if (gated && (!w->gate_codes || !w->gate_scales || !w->gate_global)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(c.hidden, c.inter, c.n_experts, c.top_k);
  if (st != MOE_OK) return st;
  if (c.max_tokens < 0) return MOE_ERR_INVALID_ARG;
  if ((long long)c.max_tokens * c.top_k > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !is_sm103(dev)) return MOE_ERR_NO_DEVICE;

  moe_nvfp4* h = new (std::nothrow) moe_nvfp4();
  if (!h) return MOE_ERR_CUDA;
  h->cfg = c;
  h->device = dev;
  h->num_sms = device_sms(dev);
  h->threshold = c.gemv_max_rows > 0 ? c.gemv_max_rows : 8;
  h->single_max_tokens = c.single_max_tokens == 0 ? kDecMaxTokens : c.single_max_tokens;
  const size_t H = c.hidden, I = c.inter, E = c.n_experts;
  const size_t R = (size_t)c.max_tokens * c.top_k, Rr = R > 0 ? R : 1;
  const size_t mat_codes = E * H * I / 2, mat_scales = E * H * I / 16;
  const size_t up_rows = gated ? 2 * I : I;  // rows of the (fused) up matrix the kernels stream
  uint8_t* gu = nullptr;                     // gated: gate and up interleaved by 16 rows, [E][2I][H/2 + H/16]
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  h->gated = gated;
#define TRY(x)                  \
  do {                          \
    e = (x);                    \
    if (e != cudaSuccess) goto fail; \
  } while (0)
  TRY(cudaMalloc(&h->up_codes, mat_codes));
  TRY(cudaMalloc(&h->dn_codes, mat_codes));
  TRY(cudaMalloc(&h->up_scales, mat_scales));
  TRY(cudaMalloc(&h->dn_scales, mat_scales));
  TRY(cudaMalloc(&h->up_g, E * sizeof(float)));
  TRY(cudaMalloc(&h->dn_g, E * sizeof(float)));
  TRY(cudaMalloc(&h->counts, E * sizeof(int32_t)));
  TRY(cudaMalloc(&h->offsets, (E + 1) * sizeof(int32_t)));
  TRY(cudaMalloc(&h->perm_pair, Rr * sizeof(int32_t)));
  TRY(cudaMalloc(&h->inv, Rr * sizeof(int32_t)));
  TRY(cudaMalloc(&h->err, sizeof(int32_t)));
  TRY(cudaMalloc(&h->blk_hist, (routing_scratch_ints((int64_t)Rr, (int)E) + 1) * sizeof(int32_t)));
  TRY(cudaMalloc(&h->Xp, Rr * H * 2));
  TRY(cudaMalloc(&h->Ap, Rr * I * 2));
  TRY(cudaMalloc(&h->Yp, Rr * H * 4));
  TRY(cudaMalloc(&h->x_stage, (size_t)(c.max_tokens > 0 ? c.max_tokens : 1) * H * 2));
  TRY(cudaMalloc(&h->dst_stage, (size_t)(c.max_tokens > 0 ? c.max_tokens : 1) * H * 2));
  TRY(cudaMalloc(&h->ids_stage, Rr * sizeof(int32_t)));
  TRY(cudaMalloc(&h->w_stage, Rr * sizeof(float)));
  TRY(cudaMalloc(&h->small_dev, kSmallStage));
  if (cudaMallocHost(&h->small_host, kSmallStage) != cudaSuccess) {
    h->small_host = nullptr;  // host calls then copy each array on its own
    cudaGetLastError();
  } else if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->small_host_dev), h->small_host, 0) !=
             cudaSuccess) {
    h->small_host_dev = nullptr;  // not mapped: the result comes back by copy
    cudaGetLastError();
  }
  if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->dst_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->part_done[0], cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->part_done[1], cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->part_done[2], cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->part_done[3], cudaEventDisableTiming) != cudaSuccess) {
    if (h->side) cudaStreamDestroy(h->side);
    if (h->dst_in) cudaEventDestroy(h->dst_in);
    h->side = nullptr;  // host calls then copy dst in order with the rest
    h->dst_in = nullptr;
    cudaGetLastError();
  }
  TRY(cudaMalloc(&h->up_tiles, (mat_codes + mat_scales) * (gated ? 2 : 1)));
  TRY(cudaMalloc(&h->dn_tiles, mat_codes + mat_scales));
  TRY(cudaMalloc(&h->up_tiles16, (mat_codes + mat_scales) * (gated ? 2 : 1)));
  TRY(cudaMalloc(&h->dn_tiles16, mat_codes + mat_scales));
  TRY(cudaMalloc(&h->up_blocks, gemm_blocks_bytes((int32_t)E, (int32_t)up_rows, (int32_t)H)));
  TRY(cudaMalloc(&h->dn_blocks, gemm_blocks_bytes((int32_t)E, (int32_t)H, (int32_t)I)));
  TRY(cudaMalloc(&h->col_done, (H / 16) * sizeof(int32_t)));
  TRY(cudaMalloc(&h->grid_bar, 2 * sizeof(int32_t)));
  TRY(cudaMalloc(&h->dec_partial, (size_t)h->num_sms * kDecPartialPerCta * sizeof(float4)));
  TRY(cudaMemcpyAsync(h->up_codes, w->up_codes, mat_codes, cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemcpyAsync(h->dn_codes, w->down_codes, mat_codes, cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemcpyAsync(h->up_scales, w->up_scales, mat_scales, cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemcpyAsync(h->dn_scales, w->down_scales, mat_scales, cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemcpyAsync(h->up_g, w->up_global, E * sizeof(float), cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemcpyAsync(h->dn_g, w->down_global, E * sizeof(float), cudaMemcpyDeviceToDevice, s));
  TRY(cudaMemsetAsync(h->err, 0, sizeof(int32_t), s));
  if (E == 1 && c.top_k == 1) {
    const size_t nt = c.max_tokens > 0 ? (size_t)c.max_tokens : 1;
    TRY(cudaMalloc(&h->dense_ids, nt * sizeof(int32_t)));
    TRY(cudaMalloc(&h->dense_w, nt * sizeof(float)));
    TRY(cudaMemsetAsync(h->dense_ids, 0, nt * sizeof(int32_t), s));
    std::vector<float> ones(nt, 1.0f);
    TRY(cudaMemcpyAsync(h->dense_w, ones.data(), nt * sizeof(float), cudaMemcpyHostToDevice, s));
    TRY(cudaStreamSynchronize(s));  // `ones` leaves scope
  }
  TRY(cudaMemsetAsync(h->counts, 0, E * sizeof(int32_t), s));
  TRY(cudaMemsetAsync(h->offsets, 0, (E + 1) * sizeof(int32_t), s));
  TRY(cudaMemsetAsync(h->Ap, 0, Rr * I * 2, s));
  TRY(cudaMemsetAsync(h->Yp, 0, Rr * H * 4, s));
  TRY(cudaMemsetAsync(h->col_done, 0, (H / 16) * sizeof(int32_t), s));
  TRY(cudaMemsetAsync(h->grid_bar, 0, 2 * sizeof(int32_t), s));
  if (gated) {
    TRY(cudaMalloc(&h->gate_codes, mat_codes));
    TRY(cudaMalloc(&h->gate_scales, mat_scales));
    TRY(cudaMalloc(&h->gate_g, E * sizeof(float)));
    TRY(cudaMemcpyAsync(h->gate_codes, w->gate_codes, mat_codes, cudaMemcpyDeviceToDevice, s));
    TRY(cudaMemcpyAsync(h->gate_scales, w->gate_scales, mat_scales, cudaMemcpyDeviceToDevice, s));
    TRY(cudaMemcpyAsync(h->gate_g, w->gate_global, E * sizeof(float), cudaMemcpyDeviceToDevice, s));
    // 16-row groups: [gate rows 16j..16j+15][up rows 16j..16j+15], codes then scales
    TRY(cudaMalloc(&gu, 2 * (mat_codes + mat_scales)));
    uint8_t* gu_codes = gu;
    uint8_t* gu_scales = gu + 2 * mat_codes;
    const size_t cblk = 16 * H / 2, sblk = 16 * H / 16, groups = E * I / 16;
    TRY(cudaMemcpy2DAsync(gu_codes, 2 * cblk, h->gate_codes, cblk, cblk, groups, cudaMemcpyDeviceToDevice, s));
    TRY(cudaMemcpy2DAsync(gu_codes + cblk, 2 * cblk, h->up_codes, cblk, cblk, groups, cudaMemcpyDeviceToDevice, s));
    TRY(cudaMemcpy2DAsync(gu_scales, 2 * sblk, h->gate_scales, sblk, sblk, groups, cudaMemcpyDeviceToDevice, s));
    TRY(cudaMemcpy2DAsync(gu_scales + sblk, 2 * sblk, h->up_scales, sblk, sblk, groups, cudaMemcpyDeviceToDevice,
                          s));
    TRY(launch_repack_frag(gu_codes, gu_scales, (int32_t)E, (int32_t)up_rows, (int32_t)H, h->up_tiles, s));
    TRY(launch_repack_frag16(gu_codes, gu_scales, (int32_t)E, (int32_t)up_rows, (int32_t)H, h->up_tiles16, s));
    TRY(launch_repack_gemm(gu_codes, gu_scales, (int32_t)E, (int32_t)up_rows, (int32_t)H, h->up_blocks, s));
  } else {
    TRY(launch_repack_frag(h->up_codes, h->up_scales, (int32_t)E, (int32_t)I, (int32_t)H, h->up_tiles, s));
    TRY(launch_repack_frag16(h->up_codes, h->up_scales, (int32_t)E, (int32_t)I, (int32_t)H, h->up_tiles16, s));
    TRY(launch_repack_gemm(h->up_codes, h->up_scales, (int32_t)E, (int32_t)I, (int32_t)H, h->up_blocks, s));
  }
  TRY(launch_repack_frag(h->dn_codes, h->dn_scales, (int32_t)E, (int32_t)H, (int32_t)I, h->dn_tiles, s));
  TRY(launch_repack_frag16(h->dn_codes, h->dn_scales, (int32_t)E, (int32_t)H, (int32_t)I, h->dn_tiles16, s));
  TRY(launch_repack_gemm(h->dn_codes, h->dn_scales, (int32_t)E, (int32_t)H, (int32_t)I, h->dn_blocks, s));
  TRY(make_tmap_act_rows(&h->tm_xp, h->Xp, Rr, H, kGemmTileRows));
  TRY(make_tmap_act_rows(&h->tm_ap, h->Ap, Rr, I, kGemmTileRows));
  TRY(cudaStreamSynchronize(s));
#undef TRY
  if (gu) cudaFree(gu);
  *out = h;
  return MOE_OK;
fail:
  cudaStreamSynchronize(s);
  if (gu) cudaFree(gu);
  free_handle(h);
  return MOE_ERR_CUDA;
}

moe_status moe_nvfp4_destroy(moe_nvfp4_t h) {
  if (!h) return MOE_OK;
  cudaDeviceSynchronize();
  free_handle(h);
  return MOE_OK;
}

// dst_ready (may be null): an event that must complete before anything reads
// dst (the single-launch kernel, or the WeightedRowSum of the multi-kernel path).
// *combine_left (may be null) set: the multi-kernel path stops before its
// WeightedRowSum and sets *combine_left = true, leaving it to the caller.
// dst_out (may be null): where the single-launch kernel writes the result
// (a device-visible copy of dst, e.g. mapped pinned host memory); *wrote_out
// tells whether that path ran.  Other paths update dst in place.
static moe_status forward_impl(moe_nvfp4* h, const uint16_t* x, const int32_t* ids, const float* tw, uint16_t* dst,
                               int32_t n, cudaStream_t s, cudaEvent_t dst_ready = nullptr,
                               bool* combine_left = nullptr, uint16_t* dst_out = nullptr, bool* wrote_out = nullptr) {
  const moe_nvfp4_config& c = h->cfg;
  const int32_t k = c.top_k, E = c.n_experts, H = c.hidden, I = c.inter;
  const int32_t R = n * k;
  const bool gemm = n > h->threshold;
  const bool pdl = !h->timing;
  h->last_n = n;
  cudaError_t e;
  DecodeArgs d{};
  d.up_tiles = h->up_tiles;
  d.dn_tiles = h->dn_tiles;
  d.up_tiles16 = h->up_tiles16;
  d.dn_tiles16 = h->dn_tiles16;
  d.up_g = h->up_g;
  d.dn_g = h->dn_g;
  d.gate_g = h->gate_g;
  d.gated = h->gated ? 1 : 0;
  d.x = x;
  d.ids = ids;
  d.tw = tw;
  d.dst = dst;
  d.dst_out = dst;
  d.Ap = h->Ap;
  d.Yp = h->Yp;
  d.g_counts = h->counts;
  d.g_offsets = h->offsets;
  d.g_perm = h->perm_pair;
  d.g_inv = h->inv;
  d.col_done = h->col_done;
  d.partial = h->dec_partial;
  d.grid_bar = h->grid_bar;
  d.err = h->err;
  d.n = n;
  d.H = H;
  d.I = I;
  d.E = E;
  d.k = k;
  if (n <= h->single_max_tokens && R <= kDecMaxPairs) {
    // the whole layer in one launch
    d.L = decode_layout(E, R, decode_can_stage(n, 0));
    if (d.L.warps >= 4) {
      if (dst_ready && cudaStreamWaitEvent(s, dst_ready, 0) != cudaSuccess) return MOE_ERR_CUDA;
      if (dst_out) {
        d.dst_out = dst_out;
        if (wrote_out) *wrote_out = true;
      }
      TimedLaunch tl(h, s, kKDecode);
      return cuda_status(launch_decode(d, h->num_sms, s));
    }
  }
  {
    TimedLaunch tl(h, s, kKRouting);
    e = launch_routing(ids, R, E, h->counts, h->offsets, h->perm_pair, h->inv, h->err, s, h->blk_hist);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (gemm) {
    TimedLaunch tl(h, s, kKGather);
    e = launch_gather(x, h->inv, n, k, H, R, h->Xp, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  // Experts with 0 < rows <= threshold: the same streaming kernel, fed by the
  // routing kernel's arrays (both projections in one launch); the GEMV pair
  // below is the fallback when its shared-memory plan does not fit.
  bool small_done = false;
  if (gemm) {
    d.ext = 1;
    d.max_rows = h->threshold;
    d.L = decode_layout(E, 0, true);
    if (d.L.warps >= 4) {
      TimedLaunch tl(h, s, kKSmall);
      e = launch_decode(d, h->num_sms, s);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      small_done = true;
    }
  }
  GemvArgs g{};
  g.counts = h->counts;
  g.offsets = h->offsets;
  g.perm_pair = h->perm_pair;
  g.E = E;
  g.k = k;
  g.max_rows = gemm ? h->threshold : 0;
  if (!small_done) {
    TimedLaunch tl(h, s, kKGemvUp);
    g.codes = h->up_codes;
    g.scales = h->up_scales;
    g.global = h->up_g;
    g.in = x;
    g.out = h->Ap;
    g.N = I;
    g.K = H;
    g.token_indexed = 1;
    g.relu2_bf16_out = 1;
    g.gate_codes = h->gate_codes;
    g.gate_scales = h->gate_scales;
    g.gate_global = h->gate_g;
    e = launch_gemv(g, s, pdl);
    g.gate_codes = nullptr;
    g.gate_scales = nullptr;
    g.gate_global = nullptr;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  Gemm2Args m{};
  m.counts = h->counts;
  m.offsets = h->offsets;
  m.G = E;
  m.min_rows = h->threshold;
  m.err = h->err;
  if (gemm) {
    TimedLaunch tl(h, s, kKGemmUp);
    m.blocks = h->up_blocks;
    m.global = h->up_g;
    m.N = h->gated ? 2 * I : I;
    m.K = H;
    m.out = h->Ap;
    m.epilogue = h->gated ? 2 : 1;
    m.global2 = h->gate_g;
    e = launch_gemm2(h->tm_xp, m, h->num_sms, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!small_done) {
    TimedLaunch tl(h, s, kKGemvDown);
    g.codes = h->dn_codes;
    g.scales = h->dn_scales;
    g.global = h->dn_g;
    g.in = h->Ap;
    g.out = h->Yp;
    g.N = H;
    g.K = I;
    g.token_indexed = 0;
    g.relu2_bf16_out = 0;
    e = launch_gemv(g, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (gemm) {
    TimedLaunch tl(h, s, kKGemmDown);
    m.blocks = h->dn_blocks;
    m.global = h->dn_g;
    m.N = H;
    m.K = I;
    m.out = h->Yp;
    m.epilogue = 0;
    e = launch_gemm2(h->tm_ap, m, h->num_sms, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (dst_ready && cudaStreamWaitEvent(s, dst_ready, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (combine_left) {
    *combine_left = true;
    return MOE_OK;
  }
  {
    TimedLaunch tl(h, s, kKCombine);
    e = launch_weighted_row_sum(dst, h->Yp, h->inv, tw, n, k, H, R, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_nvfp4_forward(moe_nvfp4_t h, const uint16_t* x, const int32_t* ids, const float* tw, uint16_t* dst,
                             int32_t n, moe_stream_t stream) {
  if (!h || n < 0) return MOE_ERR_INVALID_ARG;
  if (n > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (n == 0) return MOE_OK;
  if (!x || !ids || !tw || !dst) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(dst, 16) || !aligned(ids, 4) || !aligned(tw, 4)) return MOE_ERR_INVALID_ARG;
  return forward_impl(h, x, ids, tw, dst, n, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_nvfp4_shared_expert_forward(moe_nvfp4_t h, const uint16_t* x, uint16_t* dst, int32_t n,
                                           moe_stream_t stream) {
  if (!h || n < 0) return MOE_ERR_INVALID_ARG;
  if (h->cfg.n_experts != 1 || h->cfg.top_k != 1 || !h->dense_ids) return MOE_ERR_UNSUPPORTED;
  if (n > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (n == 0) return MOE_OK;
  if (!x || !dst || !aligned(x, 16) || !aligned(dst, 16)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(dst, 0, (size_t)n * h->cfg.hidden * 2, s) != cudaSuccess) return MOE_ERR_CUDA;
  return forward_impl(h, x, h->dense_ids, h->dense_w, dst, n, s);
}

moe_status moe_nvfp4_forward_host(moe_nvfp4_t h, const uint16_t* x, const int32_t* ids, const float* tw,
                                  uint16_t* dst, int32_t n, moe_stream_t stream) {
  if (!h || n < 0) return MOE_ERR_INVALID_ARG;
  if (n > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (n == 0) return MOE_OK;
  if (!x || !ids || !tw || !dst) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t H = h->cfg.hidden, R = (size_t)n * h->cfg.top_k;
  const size_t bx = (size_t)n * H * 2, bi = R * 4;
  const size_t oi = round16(bx), ow = oi + round16(bi), od = ow + round16(bi), total = od + bx;
  if (h->small_host && total <= kSmallStage) {
    // one pinned copy in instead of four; the single-launch kernel writes the
    // result straight into the mapped staging copy of dst (whose unwritten
    // elements already hold the pre-filled values), so nothing is copied out
    std::memcpy(h->small_host, x, bx);
    std::memcpy(h->small_host + oi, ids, bi);
    std::memcpy(h->small_host + ow, tw, bi);
    std::memcpy(h->small_host + od, dst, bx);
    if (cudaMemcpyAsync(h->small_dev, h->small_host, total, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    uint16_t* ddst = reinterpret_cast<uint16_t*>(h->small_dev + od);
    uint16_t* hout = h->small_host_dev ? reinterpret_cast<uint16_t*>(h->small_host_dev + od) : nullptr;
    bool wrote = false;
    const moe_status st = forward_impl(h, reinterpret_cast<const uint16_t*>(h->small_dev),
                                       reinterpret_cast<const int32_t*>(h->small_dev + oi),
                                       reinterpret_cast<const float*>(h->small_dev + ow), ddst, n, s, nullptr,
                                       nullptr, hout, &wrote);
    if (st != MOE_OK) return st;
    if (!wrote && cudaMemcpyAsync(h->small_host + od, ddst, bx, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    std::memcpy(dst, h->small_host + od, bx);
    return MOE_OK;
  }
  // ids, weights and x first (the routing and the gather need them); dst then
  // goes in on the side stream while the layer computes, and only the step
  // that reads dst waits for it (starting it after x keeps the two copies
  // from sharing the link)
  if (cudaMemcpyAsync(h->ids_stage, ids, R * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(h->w_stage, tw, R * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(h->x_stage, x, (size_t)n * H * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaEvent_t dst_ready = nullptr;
  const bool one_launch = n <= h->single_max_tokens && (int64_t)R <= kDecMaxPairs;  // reads dst from its start
  if (h->side && !one_launch) {
    if (cudaEventRecord(h->dst_in, s) != cudaSuccess || cudaStreamWaitEvent(h->side, h->dst_in, 0) != cudaSuccess ||
        cudaMemcpyAsync(h->dst_stage, dst, (size_t)n * H * 2, cudaMemcpyHostToDevice, h->side) != cudaSuccess ||
        cudaEventRecord(h->dst_in, h->side) != cudaSuccess)
      return MOE_ERR_CUDA;
    dst_ready = h->dst_in;
  } else if (cudaMemcpyAsync(h->dst_stage, dst, (size_t)n * H * 2, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  bool combine_left = false;
  moe_status st = forward_impl(h, h->x_stage, h->ids_stage, h->w_stage, h->dst_stage, n, s, dst_ready,
                               dst_ready ? &combine_left : nullptr);
  if (st != MOE_OK) return st;
  if (!combine_left) {
    if (cudaMemcpyAsync(dst, h->dst_stage, (size_t)n * H * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
  }
  // the WeightedRowSum in four token ranges; each range's rows of dst go back
  // on the side stream while the next range is combined
  const int32_t k = h->cfg.top_k;
  for (int part = 0; part < 4; ++part) {
    const int32_t t0 = (int32_t)((int64_t)n * part / 4), t1 = (int32_t)((int64_t)n * (part + 1) / 4);
    if (t1 == t0) continue;
    {
      TimedLaunch tl(h, s, kKCombine);
      if (launch_weighted_row_sum(h->dst_stage + (size_t)t0 * H, h->Yp, h->inv + (size_t)t0 * k,
                                  h->w_stage + (size_t)t0 * k, t1 - t0, k, (int32_t)H, (int32_t)R, s,
                                  !h->timing) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    if (cudaEventRecord(h->part_done[part], s) != cudaSuccess ||
        cudaStreamWaitEvent(h->side, h->part_done[part], 0) != cudaSuccess ||
        cudaMemcpyAsync(dst + (size_t)t0 * H, h->dst_stage + (size_t)t0 * H, (size_t)(t1 - t0) * H * 2,
                        cudaMemcpyDeviceToHost, h->side) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaStreamSynchronize(h->side) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

moe_status moe_nvfp4_get_device_error(moe_nvfp4_t h, int32_t* flags) {
  if (!h || !flags) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, h->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & MOE_DEVFLAG_TIMEOUT) {  // a wait gave up: the cross-CTA counters may be left mid-count
    if (cudaMemset(h->col_done, 0, (h->cfg.hidden / 16) * sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(h->grid_bar, 0, 2 * sizeof(int32_t)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  *flags = v;
  return MOE_OK;
}

moe_status moe_nvfp4_debug_routing(moe_nvfp4_t h, int32_t* counts, int32_t* offsets, int32_t* perm_pair,
                                   int32_t* inv, moe_stream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t E = h->cfg.n_experts, R = (size_t)h->last_n * h->cfg.top_k;
  cudaError_t e = cudaSuccess;
  if (counts && e == cudaSuccess) e = cudaMemcpyAsync(counts, h->counts, E * 4, cudaMemcpyDeviceToDevice, s);
  if (offsets && e == cudaSuccess)
    e = cudaMemcpyAsync(offsets, h->offsets, (E + 1) * 4, cudaMemcpyDeviceToDevice, s);
  if (perm_pair && R && e == cudaSuccess)
    e = cudaMemcpyAsync(perm_pair, h->perm_pair, R * 4, cudaMemcpyDeviceToDevice, s);
  if (inv && R && e == cudaSuccess) e = cudaMemcpyAsync(inv, h->inv, R * 4, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

moe_status moe_nvfp4_debug_intermediates(moe_nvfp4_t h, uint16_t* a_rows, float* y_rows, moe_stream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t R = (size_t)h->last_n * h->cfg.top_k;
  cudaError_t e = cudaSuccess;
  if (a_rows && R) e = cudaMemcpyAsync(a_rows, h->Ap, R * h->cfg.inter * 2, cudaMemcpyDeviceToDevice, s);
  if (y_rows && R && e == cudaSuccess)
    e = cudaMemcpyAsync(y_rows, h->Yp, R * h->cfg.hidden * 4, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

moe_status moe_nvfp4_debug_offset_grid_barrier(moe_nvfp4_t h, int64_t arrivals) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  uint64_t count = 0;
  if (cudaMemcpy(&count, h->grid_bar, sizeof(count), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  count += (uint64_t)arrivals;
  if (cudaMemcpy(h->grid_bar, &count, sizeof(count), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_nvfp4_set_timing(moe_nvfp4_t h, int32_t enable) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (enable && h->slots.empty()) {
    h->slots.resize(512);
    for (auto& sl : h->slots) {
      if (cudaEventCreate(&sl.beg) != cudaSuccess || cudaEventCreate(&sl.end) != cudaSuccess) return MOE_ERR_CUDA;
    }
  }
  h->timing = enable != 0;
  return MOE_OK;
}

moe_status moe_nvfp4_kernel_times(moe_nvfp4_t h, const char** names, double* total_ms, int64_t* launches,
                                  int32_t capacity, int32_t* count) {
  if (!h || !count) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  for (auto& sl : h->slots) {
    if (sl.kernel < 0) continue;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, sl.beg, sl.end) == cudaSuccess) {
      h->total_ms[sl.kernel] += ms;
      h->launches[sl.kernel] += 1;
    }
    sl.kernel = -1;
  }
  *count = kKCount;
  for (int i = 0; i < kKCount && i < capacity; ++i) {
    if (names) names[i] = kKernelNames[i];
    if (total_ms) total_ms[i] = h->total_ms[i];
    if (launches) launches[i] = h->launches[i];
  }
  for (int i = 0; i < kKCount; ++i) {
    h->total_ms[i] = 0;
    h->launches[i] = 0;
  }
  return MOE_OK;
}

moe_status nvfp4_matmul(const uint16_t* A, const uint8_t* codes, const uint8_t* scales, float global, void* C,
                        int32_t M, int32_t N, int32_t K, int32_t epilogue, moe_stream_t stream) {
  if (M < 0 || N <= 0 || K <= 0 || (epilogue != 0 && epilogue != 1)) return MOE_ERR_INVALID_ARG;
  if (K % 64 || N % 16) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (!A || !codes || !scales || !C) return MOE_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(C, 16)) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !is_sm103(dev)) return MOE_ERR_NO_DEVICE;
  CUtensorMap ta, tb;
  if (make_tmap_act(&ta, A, (uint64_t)M, (uint64_t)K) != cudaSuccess) return MOE_ERR_CUDA;
  if (make_tmap_codes(&tb, codes, (uint64_t)N, (uint64_t)K) != cudaSuccess) return MOE_ERR_CUDA;
  GemmArgs m{};
  m.scales = scales;
  m.global = nullptr;
  m.alpha0 = global;
  m.counts = nullptr;
  m.offsets = nullptr;
  m.M = M;
  m.G = 1;
  m.N = N;
  m.K = K;
  m.min_rows = 0;
  m.out = C;
  m.epilogue = epilogue;
  m.err = nullptr;
  return cuda_status(launch_gemm(ta, tb, m, device_sms(dev), reinterpret_cast<cudaStream_t>(stream), false));
}

moe_status moe_router_topk(const float* logits, const float* bias, int32_t n, int32_t n_experts, int32_t top_k,
                           int32_t* topk_ids, float* topk_weights, int32_t* counts, moe_stream_t stream) {
  if (n < 0 || n_experts <= 0 || top_k < 1 || top_k > n_experts) return MOE_ERR_INVALID_ARG;
  if (top_k > 32 || n_experts > 1024) return MOE_ERR_UNSUPPORTED;
  if (n > 0 && (!logits || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(bias, 4) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
      !aligned(counts, 4))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router(logits, bias, n, n_experts, top_k, topk_ids, topk_weights, counts,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

moe_status weighted_row_sum(uint16_t* dst, const float* src, const int32_t* rows, const float* w, int32_t n,
                            int32_t k, int32_t cols, int32_t src_rows, moe_stream_t stream) {
  if (n < 0 || k <= 0 || cols <= 0 || src_rows < 0) return MOE_ERR_INVALID_ARG;
  if (cols % 8) return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (!dst || !src || !rows || !w) return MOE_ERR_INVALID_ARG;
  if (!aligned(dst, 16) || !aligned(src, 16) || !aligned(rows, 4) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_weighted_row_sum(dst, src, rows, w, n, k, cols, src_rows, reinterpret_cast<cudaStream_t>(stream), false));
}

}  // extern "C"
