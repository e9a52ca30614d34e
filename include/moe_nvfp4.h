/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4, the NVFP4 MoE expert layer for one
 * GB300 GPU (sm_103a).
 *
 * The layer (gllm pull request #91, "perf: gather tokens per MoE expert, run
 * large NVFP4 GEMMs on bf16 tensor cores", section "What changes"): given bf16
 * activations x[n][H] and a top-k routing (ids, weights), every (token t,
 * slot j) pair p = t*k + j with expert e = ids[t][j] gets one row of a packed
 * buffer grouped by expert; each expert runs up -> relu^2 -> down over only its
 * own rows; a fixed-order weighted row sum then adds each token's k results
 * onto the pre-filled dst:
 *
 *     h      = g_up[e]   * (W_up[e]   . x[t])             fp32 accumulate
 *     a      = bf16_rne(max(h, 0)^2)                      one rounding
 *     y      = g_down[e] * (W_down[e] . a)                fp32 result
 *     dst[t] = bf16_rne(dst[t] + sum_{j=0..k-1} w[t][j] * y_(t,j))   j in order
 *
 * Gated experts (config.activation = MOE_ACT_SWIGLU; the "gate-up" expert
 * kernel of "nvfp4 experts cuda: decode kernels stall on load latency ...
 * #2265", section "What ncu shows", whose output needs both a gate row and an
 * up row; the activation is read as SwiGLU) replace the relu^2 step by
 *
 *     g      = g_gate[e] * (W_gate[e] . x[t])             fp32 accumulate
 *     a      = bf16_rne(silu(g) * h),  silu(g) = g / (1 + exp(-g))
 *
 * NVFP4 weights: W[r][c] = e2m1(code[r][c]) * e4m3(scale[r][c/16]); the
 * per-matrix fp32 global g is applied to the product (the GEMM alpha), never
 * folded into the bf16 weights (same page, bf16 NVFP4 GEMM).  Every product
 * W * x is formed exactly: the weights are unpacked without rounding to bf16,
 * or, where the small-batch kernel stages its activation rows (every expert
 * holding at most 8 tokens), to f16 against activation rows rescaled by a
 * power of two per row (exact for every value within 2^28 of its row's
 * largest magnitude); the scale is undone on the fp32 sum.
 *
 * Conventions for every entry point:
 *   - All array arguments are plain pointers.  "device" means memory the GPU
 *     can address (cudaMalloc'd); "host" means ordinary or pinned CPU memory.
 *   - bf16 arrays are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls that
 *     take a stream only enqueue work on it and return without waiting unless
 *     documented otherwise.
 *   - Matrices are row-major.  Weights are [out][in] with K (= in) contiguous:
 *       up   codes [E][I][H/2]  scales [E][I][H/16]
 *       down codes [E][H][I/2]  scales [E][H][I/16]
 *       gate codes [E][I][H/2]  scales [E][I][H/16]   (gated experts only)
 *     Code byte i of a row holds element 2i in its low nibble and element
 *     2i+1 in its high nibble.  Scale bytes are E4M3FN; NaN bytes (0x7F,
 *     0xFF) are outside the contract.
 *   - Errors: a call that returns anything but MOE_OK has enqueued nothing.
 *     Problems only the GPU can see (an expert id outside [0, E)) set a
 *     flag in handle-owned device memory; read it with
 *     moe_nvfp4_get_device_error.  No entry point aborts, traps or throws.
 *   - Shapes supported: H and I multiples of 64, 1 <= k <= 32,
 *     1 <= E <= 1024, n <= max_tokens given at create time.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum value */
  MOE_ERR_UNSUPPORTED = 2, /* a shape outside the supported set (see above) */
  MOE_ERR_CAPACITY = 3,    /* n_tokens > max_tokens of the handle */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MOE_ERR_BAD_ROUTING = 5, /* device flag: an id outside [0, E) was dropped */
  MOE_ERR_TIMEOUT = 6,     /* device flag: a bounded in-kernel wait ran out */
  MOE_ERR_NO_DEVICE = 7    /* no usable sm_103 device */
} moe_status;

/* Device error flag bits reported by moe_nvfp4_get_device_error. */
#define MOE_DEVFLAG_BAD_ROUTING 0x1
#define MOE_DEVFLAG_TIMEOUT 0x2

typedef void *moe_stream_t; /* a cudaStream_t */

typedef struct moe_nvfp4 *moe_nvfp4_t;

/* Expert activation (moe_nvfp4_config.activation). */
#define MOE_ACT_RELU2 0  /* a = bf16(max(h, 0)^2) */
#define MOE_ACT_SWIGLU 1 /* a = bf16(silu(g) * h), gate weights required */

typedef struct moe_nvfp4_config {
  int32_t hidden;        /* H */
  int32_t inter;         /* I, the expert intermediate size */
  int32_t n_experts;     /* E */
  int32_t top_k;         /* k */
  int32_t max_tokens;    /* largest n a forward may be called with */
  int32_t gemv_max_rows; /* in a batch that is not run as one launch (see
                            moe_nvfp4_forward), experts with at most this many
                            rows take the weight-streaming path, larger ones
                            the tensor-core grouped GEMM; <= 0 selects 8 (pull
                            request #91, "Results", uses 32 for its GEMV; 8 is
                            the measured best here for the 4314-token
                            prefill) */
  int32_t single_max_tokens; /* batches with n <= this and n * k <= 1024 run
                                as one launch; 0 selects 64, < 0 never */
  int32_t activation;        /* MOE_ACT_RELU2 (0) or MOE_ACT_SWIGLU (1) */
} moe_nvfp4_config;

typedef struct moe_nvfp4_weights { /* device pointers, layouts as above */
  const uint8_t *up_codes;
  const uint8_t *up_scales;
  const uint8_t *down_codes;
  const uint8_t *down_scales;
  const float *up_global;   /* [E] */
  const float *down_global; /* [E] */
  const uint8_t *gate_codes;  /* MOE_ACT_SWIGLU: [E][I][H/2]; otherwise ignored (may be NULL) */
  const uint8_t *gate_scales; /* MOE_ACT_SWIGLU: [E][I][H/16] */
  const float *gate_global;   /* MOE_ACT_SWIGLU: [E] */
} moe_nvfp4_weights;

/* Human-readable name of a status (static storage, never NULL). */
MOE_API const char *moe_nvfp4_status_string(moe_status status);

/* Create a layer on the current CUDA device.
 * Copies the weights into library-owned device memory (the caller may free
 * its copies once this returns) and allocates the whole workspace for
 * max_tokens, so that forward never allocates (pull request #91, "Results",
 * names per-op cudaMalloc/cudaFree as the remaining host cost).  Work is
 * enqueued on `stream`, which is synchronized before returning.
 * Errors: MOE_ERR_INVALID_ARG (null pointer -- the gate arrays too when
 * activation is MOE_ACT_SWIGLU --, max_tokens < 0, activation not one of the
 * MOE_ACT_ values), MOE_ERR_UNSUPPORTED (shape), MOE_ERR_NO_DEVICE,
 * MOE_ERR_CUDA (allocation).
 * On error *out is set to NULL and nothing stays allocated. */
MOE_API moe_status moe_nvfp4_create(const moe_nvfp4_config *config, const moe_nvfp4_weights *weights,
                            moe_stream_t stream, moe_nvfp4_t *out);

/* Free everything the handle owns (synchronizes the device first).  NULL is a no-op. */
MOE_API moe_status moe_nvfp4_destroy(moe_nvfp4_t handle);

/* The layer on device buffers (see top of file for the arithmetic).
 *   x            device bf16 [n][H]
 *   topk_ids     device int32 [n][k]
 *   topk_weights device fp32 [n][k], used as given (no renormalisation)
 *   dst          device bf16 [n][H], read and updated in place
 * A batch with n <= single_max_tokens (default 64) and n * k <= 1024 runs as
 * one cooperative launch
 * (routing, both projections and the combine in one kernel, one CTA per SM);
 * a larger one enqueues the routing, the gather, the streaming kernel for
 * experts with at most gemv_max_rows rows, the tensor-core grouped GEMMs and
 * the combine on `stream`.  No host synchronisation, no allocation, no host
 * read of device data.  A handle's workspace serves one forward at a time: calls on one
 * stream are ordered; concurrent streams need separate handles.  n = 0
 * returns MOE_OK and enqueues nothing.  Results are bitwise deterministic for
 * a given handle configuration.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CAPACITY (n > max_tokens), MOE_ERR_CUDA. */
MOE_API moe_status moe_nvfp4_forward(moe_nvfp4_t handle, const uint16_t *x, const int32_t *topk_ids,
                             const float *topk_weights, uint16_t *dst, int32_t n_tokens,
                             moe_stream_t stream);

/* Same layer on HOST buffers (pinned memory gives full copy speed): copies
 * x, ids, weights and dst to handle-owned device staging buffers, runs the
 * forward, copies dst back and synchronizes `stream` before returning.  When
 * the four inputs total at most 64 KB (decode-sized batches) they are first
 * packed on the host into one handle-owned pinned buffer, so one copy moves
 * them in; when that batch runs as the single launch, the kernel writes the
 * result straight into the buffer's device-mapped dst copy (no copy out),
 * otherwise one copy moves dst out.  Larger calls copy dst in on a handle-owned
 * side stream while the layer computes (only the step that reads dst waits
 * for that copy), and on the multi-kernel path the result comes back in four
 * token ranges, each copied out while the next is combined.
 * Same arguments and errors as moe_nvfp4_forward. */
MOE_API moe_status moe_nvfp4_forward_host(moe_nvfp4_t handle, const uint16_t *x_host, const int32_t *topk_ids_host,
                                  const float *topk_weights_host, uint16_t *dst_host, int32_t n_tokens,
                                  moe_stream_t stream);

/* The shared expert: the same expert FFN applied to every token with weight 1,
 * WRITING its output to dst (the pre-filled dst that moe_nvfp4_forward adds
 * the routed experts onto; pull request #91, "What changes", WeightedRowSum
 * "onto the shared expert's" output):
 *     dst[t] = bf16_rne(y(x[t]))      y as at the top of the file, expert 0
 * The handle must have been created with n_experts = 1 and top_k = 1 (its
 * weights are the shared expert's); it runs the same kernels as
 * moe_nvfp4_forward, with every token routed to expert 0 at weight 1 onto a
 * zeroed dst.  x device bf16 [n][H], dst device bf16 [n][H] (written).
 * Enqueues a memset of dst and the forward on `stream`; capturable in the same
 * CUDA graph as the routed layer's forward that follows it.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (handle not 1 expert,
 * top-1), MOE_ERR_CAPACITY, MOE_ERR_CUDA. */
MOE_API moe_status moe_nvfp4_shared_expert_forward(moe_nvfp4_t handle, const uint16_t *x, uint16_t *dst,
                                                   int32_t n_tokens, moe_stream_t stream);

/* Reads and clears the handle's device error flags (MOE_DEVFLAG_* bits).
 * Synchronizes the device. */
MOE_API moe_status moe_nvfp4_get_device_error(moe_nvfp4_t handle, int32_t *flags);

/* Copies the routing of the most recent forward into caller device buffers
 * (any pointer may be NULL to skip it), ordered on `stream`:
 *   counts [E], offsets [E+1], perm_pair [n*k] (pair index p of packed row r),
 *   inv [n*k] (packed row of pair p, -1 for a dropped pair).
 * Rows of one expert are in ascending pair order. */
MOE_API moe_status moe_nvfp4_debug_routing(moe_nvfp4_t handle, int32_t *counts, int32_t *offsets, int32_t *perm_pair,
                                   int32_t *inv, moe_stream_t stream);

/* Copies the packed per-row intermediates of the most recent forward into
 * caller device buffers (NULL skips): a_rows bf16 [n*k][I] (relu^2 output),
 * y_rows fp32 [n*k][H] (down projection), ordered on `stream`. */
MOE_API moe_status moe_nvfp4_debug_intermediates(moe_nvfp4_t handle, uint16_t *a_rows, float *y_rows,
                                         moe_stream_t stream);

/* Test hook for the failure path: adds `arrivals` to the arrival count of the
 * streaming kernel's grid barrier (synchronizes the device).  A count that is
 * no longer a multiple of the grid makes the next single-launch forward's
 * barrier unable to complete for some CTAs: their bounded wait gives up after
 * about 2 s, sets MOE_DEVFLAG_TIMEOUT and the launch returns (its output is
 * then undefined); moe_nvfp4_get_device_error reports the flag and resets the
 * counters, after which forwards are correct again.  No fault, trap or hang
 * is involved.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
MOE_API moe_status moe_nvfp4_debug_offset_grid_barrier(moe_nvfp4_t handle, int64_t arrivals);

/* Per-kernel CUDA-event timing of forward (off by default).  While on, each
 * kernel launch of forward is bracketed by an event pair on its stream. */
MOE_API moe_status moe_nvfp4_set_timing(moe_nvfp4_t handle, int32_t enable);

/* Accumulated per-kernel times since timing was enabled (synchronizes).
 * Fills up to `capacity` entries: names[i] (static strings), total_ms[i] and
 * launches[i]; *count receives the number of kernels seen.  Resets the sums. */
MOE_API moe_status moe_nvfp4_kernel_times(moe_nvfp4_t handle, const char **names, double *total_ms, int64_t *launches,
                                  int32_t capacity, int32_t *count);

/* Dense NVFP4 GEMM on the tensor cores (pull request #91, "What changes",
 * bf16 NVFP4 GEMM; "Testing", TestCUDAMatMulNVFP4Exact):
 *   C[m][j] = global * sum_c A[m][c] * W[j][c]
 *   A       device bf16 [M][K]
 *   codes   device u8 [N][K/2], scales device u8 [N][K/16] (layout as above)
 *   C       device, epilogue 0: fp32 [M][N];
 *                   epilogue 1: bf16 [M][N] holding bf16_rne(max(C, 0)^2)
 * K must be a multiple of 64 and N of 16; M >= 0 (M = 0 enqueues nothing).
 * The weights are unpacked exactly to bf16 in shared memory and fed to
 * tcgen05 MMAs with fp32 accumulation in tensor memory.  Allocates nothing.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API moe_status nvfp4_matmul(const uint16_t *A, const uint8_t *codes, const uint8_t *scales, float global, void *C,
                        int32_t M, int32_t N, int32_t K, int32_t epilogue, moe_stream_t stream);

/* The router that produces the layer's topk_ids / topk_weights (the step
 * before the layer; the layer's workloads are routed this way: fp32 logits,
 * optionally plus a per-expert bias, top-k, softmax renormalised over the k
 * picked).  For each token t:
 *   z[e]            = logits[t][e] + bias[e]   (one fp32 addition; bias may be NULL)
 *   topk_ids[t]     = the top_k experts by descending z, equal z lower index first
 *   topk_weights[t] = exp(z_j - z_0) / sum_i exp(z_i - z_0) over the picks (fp32)
 *   counts[e]       = tokens that picked e (optional, may be NULL; zeroed first)
 *   logits device fp32 [n][n_experts], bias device fp32 [n_experts],
 *   topk_ids device int32 [n][top_k], topk_weights device fp32 [n][top_k],
 *   counts device int32 [n_experts].
 * One warp per token; ids are exact (fp32 comparisons), weights run-to-run
 * identical.  Enqueued on `stream`, no allocation.  NaN logits are outside
 * the contract.  Errors: MOE_ERR_INVALID_ARG (n < 0, top_k outside
 * [1, n_experts], null or misaligned pointer), MOE_ERR_UNSUPPORTED
 * (top_k > 32 or n_experts > 1024), MOE_ERR_CUDA. */
MOE_API moe_status moe_router_topk(const float *logits, const float *bias, int32_t n, int32_t n_experts,
                                   int32_t top_k, int32_t *topk_ids, float *topk_weights, int32_t *counts,
                                   moe_stream_t stream);

/* Deterministic weighted row sum (pull request #91, "What changes",
 * WeightedRowSum):
 *   dst[i][c] = bf16_rne(dst[i][c] + sum_{j=0..k-1} w[i][j] * src[rows[i][j]][c])
 * with the j terms added in increasing order by one fp32 fused multiply-add
 * each, one thread per output element, no atomics.
 *   dst device bf16 [n][cols] (in place), src device fp32 [src_rows][cols],
 *   rows device int32 [n][k], w device fp32 [n][k].
 * A row index outside [0, src_rows) contributes nothing.  cols must be a
 * multiple of 8.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API moe_status weighted_row_sum(uint16_t *dst, const float *src, const int32_t *rows, const float *w, int32_t n,
                            int32_t k, int32_t cols, int32_t src_rows, moe_stream_t stream);

/* The layer for callers that cannot allocate device memory.  The pages have
 * no counterpart of this call.  Some callers cannot call cudaMalloc: a plugin
 * or server whose host process owns all device memory through its own pool
 * and must account for every byte, a caller with a memory budget fixed at
 * load time, or code that must not risk the device-wide synchronisation an
 * allocation can cause.  This call needs no handle and allocates nothing:
 *   config, weights  as for moe_nvfp4_create, but the weights are read in
 *                    place from the caller's device memory on every call
 *   x, topk_ids, topk_weights, dst, n_tokens, stream  as for moe_nvfp4_forward
 * Every intermediate (routing arrays, relu^2 rows, down rows, error flag)
 * lives in one file-scope device array of 8 MiB that every GPU which loads
 * the library holds until the process exits.  A call needs
 *   about 4*(2E + 2R) + R*(2*I + 4*H) bytes of it, R = n_tokens * top_k
 * (for H = 2688, I = 1856, E = 128 that is up to 579 rows, 96 tokens at
 * top-6); larger calls return
 * MOE_ERR_CAPACITY and enqueue nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) and caches it: make that
 * first call before any stream capture.  All calls on a device share the
 * array and it keeps the last call's contents, so calls whose work overlaps
 * on the GPU race on it; order them.  Every expert runs on the weight-
 * streaming kernel; ids outside [0, E) are dropped (they add nothing) and
 * are not reported.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_CAPACITY, MOE_ERR_NO_DEVICE, MOE_ERR_CUDA. */
MOE_API moe_status moe_nvfp4_forward_noalloc(const moe_nvfp4_config *config, const moe_nvfp4_weights *weights,
                                             const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                                             uint16_t *dst, int32_t n_tokens, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
