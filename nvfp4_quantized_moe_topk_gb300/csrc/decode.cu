// decode.cu -- the whole layer in one persistent launch for small batches.
//
// At one token the layer reads 6 experts x 5.6 MB of NVFP4 weights and almost
// nothing else, so its time is set by how early and how fast those bytes
// stream in.  TensorFold issue #2265 ("Proposal") finds such decode kernels
// stalled on load latency and keeps, per warp, a ring of shared-memory stages
// filled asynchronously with the weight words, block scales and input rows;
// gllm pull request #91 ("Results") runs experts holding at most 32 tokens on
// a GEMV.  Here one cooperative kernel (one CTA per SM) does the whole layer:
//
//   1. warp 0 routes the <= 1024 pairs in shared memory (counts, offsets,
//      stable permutation), identically in every CTA;
//   2. the CTA's share of (expert, 16-row tile) items -- up tiles, then down
//      tiles; two consecutive row tiles per item once an expert holds two or
//      more tokens -- is laid out as one run of 64-wide k-tiles per phase and
//      cut evenly over the warps (a warp's range may start or end inside an
//      item);
//   3. each warp streams its range through a private ring of slots; a slot
//      holds a chunk of up to 4 weight k-tiles and the matching activation row
//      segments of up to 8 tokens, all copied by 1-D bulk copies completing on
//      the slot's mbarrier, several chunks ahead of use; no warp waits on
//      another in the loop;
//   4. the warp unpacks its codes exactly to bf16 in registers (bit placement
//      + one bf16 multiply by the e4m3 scale, see below) and feeds them as A
//      fragments of warp-level bf16 MMAs with fp32 accumulation; the last warp
//      holding part of a tile sums the parts in warp order and writes it:
//      relu^2 + bf16 rounding fused into the up store, fp32 rows for down;
//      a gated expert's up item is its gate tile and its up tile of the same
//      16 rows (the TensorFold gate-up kernel's "both rows"), and the store
//      is bf16(silu(gate) * up);
//   5. one grid barrier (a single arrival per CTA) separates up from down; the
//      weight chunks of the first down tiles are already in flight across it,
//      their activation rows (the relu^2 rows) are requested right after it;
//   6. the WeightedRowSum onto dst (j ascending, one fma each, no atomics on
//      data): for up to 8 tokens the last warp to finish a 16-column block of
//      down tiles applies it to those columns, for more tokens every thread
//      takes one element after a second grid barrier.
//
// The same kernel also serves the experts with few rows inside a large batch
// (external-routing mode): it then takes the counts, offsets and permutation
// that the routing kernel wrote, works only on experts whose row count is at
// most the GEMV threshold, and leaves the combine to the WeightedRowSum
// kernel that runs after the grouped GEMMs.
//
// Fragment-tile weight layout (written once at create): a matrix [G][N][K]
// becomes tiles [G][N/16][K/64] of 576 bytes -- 512 code bytes, 16 B per lane,
// then the 16 rows x 4 e4m3 scales.  Within a tile the k order seen by the MMA
// is permuted so that lane (g = l/4, t = l%4) owns the 16 consecutive k
// 16t .. 16t+15 of rows g and g+8: that is exactly one scale block per row, and
// the activation bytes it multiplies are 32 contiguous bytes.  The same
// permutation is applied to the activations simply by where each lane loads
// them from, so the MMA sums the right products.  The 8 codes of one 32-bit
// word are bit-placed so that each bf16 pair of the A fragment is one or two
// shifts and one mask away: a code lands as sign|exponent(2)|mantissa(1) in the
// bf16 sign / low exponent / top mantissa bits, i.e. as e2m1 * 2^-126, and one
// bf16 multiply by (e4m3 scale * 2^118) gives the exact weight * 2^-8, undone
// by scaling alpha by 2^8.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------------ repack
__global__ void repack_frag_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                   int32_t G, int32_t N, int32_t K, uint8_t* __restrict__ out) {
  const int32_t KT = K / 64, NT = N / 16;
  const long long tiles = (long long)G * NT * KT;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < tiles * 32;
       i += (long long)gridDim.x * blockDim.x) {
    const long long tile = i >> 5;
    const int lane = (int)(i & 31);
    const int kt = (int)(tile % KT);
    const long long rest = tile / KT;
    const int rt = (int)(rest % NT);
    const long long grp = rest / NT;
    const int g = lane >> 2, t = lane & 3;
    uint32_t words[4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const long long row = grp * N + rt * 16 + g + 8 * half;
      // the lane's 16 codes of this row: k = 64 kt + 16 t .. +15 = 8 code bytes
      const uint8_t* src = codes + row * (K / 2) + kt * 32 + 8 * t;
#pragma unroll
      for (int wq = 0; wq < 2; ++wq) {
        uint32_t w = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // pair slot p of this word = code byte 4 wq + p
          const uint32_t byte = src[4 * wq + p];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t code = (byte >> (4 * h)) & 15u;
#pragma unroll
            for (int b = 0; b < 4; ++b) w |= ((code >> b) & 1u) << code_bit_pos(p, h, b);
          }
        }
        words[2 * half + wq] = w;
      }
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + tile * kTileBytes + 16 * lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = words[q];
    if (lane < 16) {
      const long long row = grp * N + rt * 16 + lane;
      uint8_t* sd = out + tile * kTileBytes + 512 + 4 * lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) sd[j] = scales[row * (K / 16) + kt * 4 + j];
    }
  }
}

cudaError_t launch_repack_frag(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                               uint8_t* out, cudaStream_t s) {
  const long long work = (long long)G * (N / 16) * (K / 64) * 32;
  long long blocks = (work + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  if (blocks < 1) blocks = 1;
  repack_frag_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, scales, G, N, K, out);
  return cudaGetLastError();
}

// Byte-order fragment tiles for the f16 path: the same [G][N/16][K/64] tiles
// of 576 bytes and the same scale bytes, but lane (g, t)'s 16 code bytes are
// whole NVFP4 bytes (two consecutive k, the lower k in the low nibble), in the
// order the f16 MMA takes them.  Word j serves MMA j of the k-tile, which sums
// k = 16t + 4j .. 16t + 4j + 3 of this lane (the lane's 16 consecutive k are
// still one scale block per row): bytes [row g, k 16t+4j..+1], [row g+8, the
// same], [row g, k 16t+4j+2..+3], [row g+8, the same] = A registers a0..a3.
__global__ void repack_frag16_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                     int32_t G, int32_t N, int32_t K, uint8_t* __restrict__ out) {
  const int32_t KT = K / 64, NT = N / 16;
  const long long tiles = (long long)G * NT * KT;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < tiles * 32;
       i += (long long)gridDim.x * blockDim.x) {
    const long long tile = i >> 5;
    const int lane = (int)(i & 31);
    const int kt = (int)(tile % KT);
    const long long rest = tile / KT;
    const int rt = (int)(rest % NT);
    const long long grp = rest / NT;
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* row0 = codes + (grp * N + rt * 16 + g) * (long long)(K / 2) + kt * 32 + 8 * t;
    const uint8_t* row8 = row0 + 8LL * (K / 2);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + tile * kTileBytes + 16 * lane);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[j] = (uint32_t)row0[2 * j] | ((uint32_t)row8[2 * j] << 8) | ((uint32_t)row0[2 * j + 1] << 16) |
               ((uint32_t)row8[2 * j + 1] << 24);
    if (lane < 16) {
      const long long row = grp * N + rt * 16 + lane;
      uint8_t* sd = out + tile * kTileBytes + 512 + 4 * lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) sd[j] = scales[row * (K / 16) + kt * 4 + j];
    }
  }
}

cudaError_t launch_repack_frag16(const uint8_t* codes, const uint8_t* scales, int32_t G, int32_t N, int32_t K,
                                 uint8_t* out, cudaStream_t s) {
  const long long work = (long long)G * (N / 16) * (K / 64) * 32;
  long long blocks = (work + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  if (blocks < 1) blocks = 1;
  repack_frag16_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, scales, G, N, K, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The four NVFP4 bytes of w as f16 pairs (hardware conversion: the low
// nibble becomes the low half), exact.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  asm("{.reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;}"
      : "=r"(p0), "=r"(p1), "=r"(p2), "=r"(p3)
      : "r"(w));
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// f16 pair (both halves) of an e4m3 byte's value, exact: |v| <= 448 and the
// smallest subnormal 2^-9 are normal f16 numbers with at most 4 significant bits.
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v = e ? (float)(8u + m) * __uint_as_float((e - 10u + 127u) << 23) : (float)m * 0x1p-9f;
  if (b & 0x80u) v = -v;
  const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(v));
  return h | (h << 16);
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t atom_add_acq_rel_gpu_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void all_warps_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ------------------------------------------------------------ work cursor
// A warp's work is a sequence of segments: k-tiles [kt, kt_end) of the
// 16-row tile rt of expert e (local item i of the phase), for tokens tok0 ..
// tok0 + 7 of that expert.  Phase 0 is the up projection, phase 1 down, 2 done.
struct __align__(16) Cur {
  int32_t ph, i, tok0, kt, kt_end, e, rt, cnt, off, srow, pad1, pad2;  // srow: first stage row (staged mode)
};

__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Ring slot layout: kDecCK weight tiles, then the chunk's activation rows:
// per token column g < nt, kDecCK x 64 bf16 (128 B per k-tile), rows padded to
// kDecActRow bytes so the 8 columns of a fragment load hit distinct banks.
constexpr uint32_t kDecActRow = kDecCK * 128 + 16;

struct DecodeCtx {
  const DecodeArgs& a;
  const int32_t* s_tok;     // packed row -> token
  const int32_t* s_counts;  // [E]
  const int32_t* s_off;     // [E+1]
  const int32_t* s_act;     // selected experts in expert order
  int32_t warp, W;
  int32_t split;            // 1: each phase's k-tiles are cut evenly over the warps (one pass of <= 8 tokens)
  int32_t u_lo, n_up, d_lo, n_dn;  // this CTA's items per phase
  int32_t KTu, KTd, NTu, NTd;
  int32_t pu, pd;           // per phase, 1: a work item is two consecutive row tiles, 0: one
  int32_t NPu, NPd;         // work items per expert
  uint32_t wbytes;          // weight bytes of a ring slot (the activation rows follow)
  int32_t Wu, Wd;           // warps that take part in each phase (split mode)
  int32_t ura, urb, dra, drb;      // this warp's tile range per phase (split mode)
  // Staged mode: the activation rows of the CTA's experts are copied once per
  // phase into a CTA-wide stage instead of with every chunk.
  int32_t staged;
  uint8_t* stage;
  uint32_t RSu, RSd;               // stage row stride per phase
  const int32_t* sbu;              // up: first stage row of staged expert j (span_u + 1 entries)
  const int32_t* sbd;              // down: the same
  int32_t elo_u, elo_d, span_u, span_d;  // first staged expert (index into s_act) and count, per phase

  __device__ DecodeCtx(const DecodeArgs& args) : a(args) {}

  template <bool S>
  __device__ __forceinline__ void load_item(Cur& c) const {
    const int32_t lo = c.ph ? d_lo : u_lo, NP = c.ph ? NPd : NPu;
    const int32_t flat = lo + c.i;
    const int32_t ei = flat / NP;
    c.rt = (flat - ei * NP) << (c.ph ? pd : pu);  // first row tile of the item
    c.e = s_act[ei];
    c.cnt = s_counts[c.e];
    c.off = s_off[c.e];
    if (S) c.srow = (c.ph ? sbd : sbu)[ei - (c.ph ? elo_d : elo_u)];
  }
  // First segment of phase ph or a later one (ph = 2 when the warp is done).
  template <bool S>
  __device__ __forceinline__ void enter_phase(Cur& c, int32_t ph) const {
    for (; ph < 2; ++ph) {
      c.ph = ph;
      c.tok0 = 0;
      const int32_t KT = ph ? KTd : KTu;
      if (warp >= W) continue;
      if (split) {
        const int32_t ra = ph ? dra : ura, rb = ph ? drb : urb;
        if (ra < rb) {
          c.i = ra / KT;
          c.kt = ra - c.i * KT;
          c.kt_end = min(KT, rb - c.i * KT);
          load_item<S>(c);
          return;
        }
      } else if (warp < (ph ? n_dn : n_up)) {
        c.i = warp;
        c.kt = 0;
        c.kt_end = KT;
        load_item<S>(c);
        return;
      }
    }
    c.ph = 2;
  }
  template <bool S>
  __device__ __forceinline__ void advance(Cur& c) const {
    c.kt += kDecCK;
    if (c.kt < c.kt_end) return;
    const int32_t KT = c.ph ? KTd : KTu;
    if (split) {
      const int32_t rb = c.ph ? drb : urb;
      ++c.i;
      if (c.i * KT < rb) {
        c.kt = 0;
        c.kt_end = min(KT, rb - c.i * KT);
        load_item<S>(c);
        return;
      }
    } else {
      c.tok0 += kDecPassTok;
      if (c.tok0 < c.cnt) {
        c.kt = 0;
        return;
      }
      c.tok0 = 0;
      c.i += W;
      if (c.i < (c.ph ? n_dn : n_up)) {
        c.kt = 0;
        load_item<S>(c);
        return;
      }
    }
    enter_phase<S>(c, c.ph + 1);
  }
  // Staged chunks stream the byte-order tiles of the f16 path.
  template <bool S>
  __device__ __forceinline__ const uint8_t* chunk_src(const Cur& c) const {
    const int32_t KT = c.ph ? KTd : KTu, NT = c.ph ? NTd : NTu;
    const uint8_t* base = S ? (c.ph ? a.dn_tiles16 : a.up_tiles16) : (c.ph ? a.dn_tiles : a.up_tiles);
    return base + ((size_t)((size_t)c.e * NT + c.rt) * KT + c.kt) * kTileBytes;
  }
  __device__ __forceinline__ int32_t kts(const Cur& c) const { return min(kDecCK, c.kt_end - c.kt); }
  __device__ __forceinline__ bool two(const Cur& c) const {
    return (c.ph ? pd : pu) && c.rt + 1 < (c.ph ? NTd : NTu);
  }
  // Lane 0 only: declare the chunk's bytes (the k-tiles of both row tiles and
  // the activation rows, the latter possibly issued later) and bulk-copy the
  // weight tiles: row tile rt into the slot's first half, rt + 1 (the next
  // KT tiles in memory) into the second.
  template <bool S>
  __device__ __forceinline__ void issue_weights(const Cur& c, uint8_t* slot, uint64_t* bar, uint64_t pol) const {
    const uint32_t n_kt = (uint32_t)kts(c);
    const uint32_t nt = (uint32_t)min(kDecPassTok, c.cnt - c.tok0);
    const bool pair = two(c);
    mbar_arrive_expect_tx(bar, n_kt * ((pair ? 2u : 1u) * kTileBytes + (S ? 0u : nt * 128u)));
    const uint8_t* src = chunk_src<S>(c);
    bulk_g2s_hint(slot, src, n_kt * kTileBytes, bar, pol);
    if (pair)
      bulk_g2s_hint(slot + kDecCK * kTileBytes, src + (size_t)(c.ph ? KTd : KTu) * kTileBytes, n_kt * kTileBytes,
                    bar, pol);
  }
  // Lanes g < nt: bulk-copy token column g's activation row segment (kts x 64
  // bf16) into the slot; it completes on the slot's barrier.
  template <bool S>
  __device__ __forceinline__ void issue_acts(const Cur& c, int lane, uint8_t* slot, uint64_t* bar) const {
    if (S) return;
    const int32_t nt = min(kDecPassTok, c.cnt - c.tok0);
    if (lane < nt) {
      const int32_t pr = c.off + c.tok0 + lane;
      const uint16_t* src;
      if (c.ph == 0) {
        const int32_t tok = a.ext ? __ldg(a.g_perm + pr) / a.k : s_tok[pr];
        src = a.x + (size_t)tok * a.H + c.kt * 64;
      } else {
        src = a.Ap + (size_t)pr * a.I + c.kt * 64;
      }
      bulk_g2s(slot + wbytes + lane * kDecActRow, src, (uint32_t)kts(c) * 128u, bar);
    }
  }
  // Lanes of one warp: copy the activation rows of phase ph's staged experts
  // into the stage (expert j's rows from stage row sb[j] on, one bulk copy
  // each) after lane 0 has declared their bytes on the stage barrier.  The
  // stage may hold the previous phase's rows, read through the generic proxy
  // by every warp before the CTA barrier that precedes this call.
  __device__ __forceinline__ void issue_stage(int32_t ph, int lane, uint64_t* bar) const {
    const int32_t* sb = ph ? sbd : sbu;
    const int32_t span = ph ? span_d : span_u, elo = ph ? elo_d : elo_u;
    const int32_t K = ph ? a.I : a.H;
    const uint32_t RS = ph ? RSd : RSu;
    const int32_t rows = span > 0 ? sb[span] : 0;
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)rows * (uint32_t)K * 2u);
    __syncwarp();
    for (int32_t r = lane; r < rows; r += 32) {
      int32_t j = 0;
      while (j + 1 < span && sb[j + 1] <= r) ++j;
      const int32_t pr = s_off[s_act[elo + j]] + (r - sb[j]);
      const uint16_t* src;
      if (ph == 0) {
        const int32_t tok = a.ext ? __ldg(a.g_perm + pr) / a.k : s_tok[pr];
        src = a.x + (size_t)tok * a.H;
      } else {
        src = a.Ap + (size_t)pr * a.I;
      }
      fence_proxy_async_smem();
      bulk_g2s(stage + (size_t)r * RS, src, (uint32_t)K * 2u, bar);
    }
  }
};

// Work items of one CTA per phase: a work item is one 16-row tile of one
// active expert, or two consecutive ones (p = 1) once some expert holds two
// or more tokens (gated: always the gate and up tiles of the same rows).
struct DecItems {
  int32_t pu, pd, NPu, NPd, u_lo, n_up, d_lo, n_dn;
};
__device__ __forceinline__ DecItems dec_items(const DecodeArgs& a, int32_t n_act, int32_t cmax) {
  DecItems it;
  it.pd = cmax >= 2;
  it.pu = it.pd || a.gated;
  const int32_t NTu = (a.gated ? 2 * a.I : a.I) / 16, NTd = a.H / 16;
  it.NPu = (NTu + it.pu) >> it.pu;
  it.NPd = (NTd + it.pd) >> it.pd;
  // n_act <= E <= 1024 and NP <= 256 (H, I <= 4096) keep U * G and D * G far below 2^32
  const uint32_t G = gridDim.x, b = blockIdx.x;
  const uint32_t U = (uint32_t)n_act * (uint32_t)it.NPu, D = (uint32_t)n_act * (uint32_t)it.NPd;
  it.u_lo = (int32_t)(U * b / G);
  it.d_lo = (int32_t)(D * b / G);
  it.n_up = (int32_t)(U * (b + 1) / G) - it.u_lo;
  it.n_dn = (int32_t)(D * (b + 1) / G) - it.d_lo;
  return it;
}

// Warp 0, after the routing: decide whether this CTA stages its activation
// rows (every expert holds at most 8 tokens, each phase's items span at most
// kDecMaxSpan experts, and the larger phase's rows fit kDecStageMax bytes)
// and write each phase's first stage row per expert.  misc[3] = staged,
// misc[4] = stage bytes, misc[5..8] = first expert and span, up then down.
__device__ __forceinline__ void decode_stage_plan(const DecodeArgs& a, int lane, const int32_t* s_counts,
                                                  const int32_t* s_act, int32_t* misc, int32_t* s_sbase) {
  __syncwarp();
  const int32_t n_act = misc[1], cmax = misc[2];
  if (cmax < 2 || cmax > kDecPassTok) {
    // one token per expert: a chunk brings one activation row segment, and
    // staging would save little against its planning on the critical path
    if (lane == 0) misc[3] = 0;
    return;
  }
  const DecItems it = dec_items(a, n_act, cmax);
  bool ok = true;
  uint32_t bytes = 0;
#pragma unroll
  for (int ph = 0; ph < 2; ++ph) {
    const int32_t lo = ph ? it.d_lo : it.u_lo, n = ph ? it.n_dn : it.n_up, NP = ph ? it.NPd : it.NPu;
    const int32_t elo = n > 0 ? lo / NP : 0;
    const int32_t span = n > 0 ? (lo + n - 1) / NP - elo + 1 : 0;
    ok = ok && span <= kDecMaxSpan;
    const int32_t c = (ok && lane < span) ? s_counts[s_act[elo + lane]] : 0;
    int32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    const int32_t rows = __shfl_sync(0xffffffffu, incl, 31);
    int32_t* sb = s_sbase + ph * (kDecMaxSpan + 1);
    if (ok && lane < span) sb[lane + 1] = incl;
    if (lane == 0) {
      sb[0] = 0;
      misc[5 + 2 * ph] = elo;
      misc[6 + 2 * ph] = ok ? span : 0;
    }
    const uint32_t need = (uint32_t)rows * (uint32_t)(2 * (ph ? a.I : a.H) + 16);
    bytes = need > bytes ? need : bytes;
  }
  bytes = (bytes + 127u) & ~127u;
  ok = ok && bytes <= (uint32_t)kDecStageMax;
  if (lane == 0) {
    misc[3] = ok;
    misc[4] = ok ? (int32_t)bytes : 0;
  }
}

// One k-tile (16 rows x 64 k) of one row tile against this lane's activation
// fragments x0 (k 16t .. 16t+7) and x1 (k 16t+8 .. 16t+15) of token column g.
__device__ __forceinline__ void tile_mma(const uint8_t* tile, const uint4& x0, const uint4& x1, int lane,
                                         const uint32_t* scale_lut, float (&acc)[4], float (&acc2)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint4 c = *reinterpret_cast<const uint4*>(tile + 16 * lane);
  const uint32_t s0 = scale_lut[tile[512 + 4 * g + t]];
  const uint32_t s1 = scale_lut[tile[512 + 4 * (g + 8) + t]];
  uint32_t r0, r1, r2, r3;  // row g
  uint32_t q0, q1, q2, q3;  // row g + 8
  // word 0 of each row: k blocks 0 and 1 of the MMA
  unpack_word(c.x, r0, r1, r2, r3);
  unpack_word(c.z, q0, q1, q2, q3);
  mma_bf16_16816(acc, mul_bf16x2(r0, s0), mul_bf16x2(q0, s1), mul_bf16x2(r1, s0), mul_bf16x2(q1, s1), x0.x, x0.y);
  mma_bf16_16816(acc2, mul_bf16x2(r2, s0), mul_bf16x2(q2, s1), mul_bf16x2(r3, s0), mul_bf16x2(q3, s1), x0.z, x0.w);
  // word 1 of each row: k blocks 2 and 3
  unpack_word(c.y, r0, r1, r2, r3);
  unpack_word(c.w, q0, q1, q2, q3);
  mma_bf16_16816(acc, mul_bf16x2(r0, s0), mul_bf16x2(q0, s1), mul_bf16x2(r1, s0), mul_bf16x2(q1, s1), x1.x, x1.y);
  mma_bf16_16816(acc2, mul_bf16x2(r2, s0), mul_bf16x2(q2, s1), mul_bf16x2(r3, s0), mul_bf16x2(q3, s1), x1.z, x1.w);
}

// One chunk: up to kDecCK k-tiles of a row-tile pair (the second only when
// `pair`) against the activation rows staged in the same slot; `act` points at
// this lane's token column.  The activation fragments of a k-tile serve both
// row tiles.
__device__ __forceinline__ void chunk_mma(const uint8_t* wts, const uint8_t* act, int kts, bool pair, int lane,
                                          const uint32_t* scale_lut, float (&accA)[4], float (&accA2)[4],
                                          float (&accB)[4], float (&accB2)[4]) {
#pragma unroll
  for (int kt = 0; kt < kDecCK; ++kt) {
    if (kt < kts) {
      const uint4 x0 = *reinterpret_cast<const uint4*>(act + kt * 128);
      const uint4 x1 = *reinterpret_cast<const uint4*>(act + kt * 128 + 16);
      tile_mma(wts + kt * kTileBytes, x0, x1, lane, scale_lut, accA, accA2);
      if (pair) tile_mma(wts + (kDecCK + kt) * kTileBytes, x0, x1, lane, scale_lut, accB, accB2);
    }
  }
}

// f16 forms of the two above, on byte-order tiles (repack_frag16_kernel) and
// f16 activation rows: word j of the lane's codes is MMA j's A fragment, each
// pair multiplied by the row's scale (f16, exact: codes have 2 and scales at
// most 4 significant bits, the product lies in [2^-10, 2688]).
__device__ __forceinline__ void tile_mma16(const uint8_t* tile, const uint4& x0, const uint4& x1, int lane,
                                           const uint32_t* lut16, float (&acc)[4], float (&acc2)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint4 c = *reinterpret_cast<const uint4*>(tile + 16 * lane);
  const uint32_t s0 = lut16[tile[512 + 4 * g + t]];
  const uint32_t s1 = lut16[tile[512 + 4 * (g + 8) + t]];
  uint32_t p0, p1, p2, p3;
  e2m1x8_to_f16(c.x, p0, p1, p2, p3);
  mma_f16_16816(acc, mul_f16x2(p0, s0), mul_f16x2(p1, s1), mul_f16x2(p2, s0), mul_f16x2(p3, s1), x0.x, x0.y);
  e2m1x8_to_f16(c.y, p0, p1, p2, p3);
  mma_f16_16816(acc2, mul_f16x2(p0, s0), mul_f16x2(p1, s1), mul_f16x2(p2, s0), mul_f16x2(p3, s1), x0.z, x0.w);
  e2m1x8_to_f16(c.z, p0, p1, p2, p3);
  mma_f16_16816(acc, mul_f16x2(p0, s0), mul_f16x2(p1, s1), mul_f16x2(p2, s0), mul_f16x2(p3, s1), x1.x, x1.y);
  e2m1x8_to_f16(c.w, p0, p1, p2, p3);
  mma_f16_16816(acc2, mul_f16x2(p0, s0), mul_f16x2(p1, s1), mul_f16x2(p2, s0), mul_f16x2(p3, s1), x1.z, x1.w);
}
__device__ __forceinline__ void chunk_mma16(const uint8_t* wts, const uint8_t* act, int kts, bool pair, int lane,
                                            const uint32_t* lut16, float (&accA)[4], float (&accA2)[4],
                                            float (&accB)[4], float (&accB2)[4]) {
#pragma unroll
  for (int kt = 0; kt < kDecCK; ++kt) {
    if (kt < kts) {
      const uint4 x0 = *reinterpret_cast<const uint4*>(act + kt * 128);
      const uint4 x1 = *reinterpret_cast<const uint4*>(act + kt * 128 + 16);
      tile_mma16(wts + kt * kTileBytes, x0, x1, lane, lut16, accA, accA2);
      if (pair) tile_mma16(wts + (kDecCK + kt) * kTileBytes, x0, x1, lane, lut16, accB, accB2);
    }
  }
}

// ------------------------------------------------------------ kernel
// Routing of all pairs by warp 0, into shared memory (every CTA computes the
// same result; CTA 0 also writes it out).  Stable: pairs of one expert keep
// increasing p order, 32 pairs at a time ranked with a warp match.
__device__ __forceinline__ void decode_route(const DecodeArgs& a, int lane, const int32_t* s_ids, int32_t* s_tok,
                                             int32_t* s_inv, const int32_t* s_counts, int32_t* s_off,
                                             int32_t* s_act, int32_t* misc) {
  const int32_t E = a.E, R = a.n * a.k;
  const int32_t per = (E + 31) / 32;
  const int32_t lo = min(E, lane * per), hi = min(E, lo + per);
  int32_t sum = 0, nact = 0, cmax = 0;
  for (int32_t e = lo; e < hi; ++e) {
    const int32_t c = s_counts[e];
    sum += c;
    nact += c > 0;
    cmax = max(cmax, c);
  }
  int32_t isum = sum, iact = nact;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t vs = __shfl_up_sync(0xffffffffu, isum, d);
    const int32_t va = __shfl_up_sync(0xffffffffu, iact, d);
    if (lane >= d) { isum += vs; iact += va; }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, d));
  int32_t run = isum - sum, ai = iact - nact;
  for (int32_t e = lo; e < hi; ++e) {
    const int32_t c = s_counts[e];
    s_off[e] = run;
    run += c;
    if (c > 0) s_act[ai++] = e;
  }
  if (lane == 31) {
    s_off[E] = isum;
    misc[1] = iact;
    misc[2] = cmax;
  }
  __syncwarp();
  const bool cta0 = blockIdx.x == 0;
  for (int32_t base = 0; base < R; base += 32) {
    const int32_t p = base + lane;
    const bool live = p < R;
    const int32_t e = live ? s_ids[p] : -1;
    const bool valid = live && e >= 0 && e < E;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int32_t rank = __popc(peers & ((1u << lane) - 1u));
    const int32_t pos = valid ? s_off[e] + rank : -1;
    __syncwarp();
    if (valid && rank == 0) s_off[e] += __popc(peers);
    __syncwarp();
    if (live) {
      s_inv[p] = pos;
      if (valid) s_tok[pos] = p / a.k;
      if (cta0) {
        a.g_inv[p] = pos;
        if (valid) a.g_perm[pos] = p;
      }
    }
  }
  __syncwarp();
  for (int32_t e = lo; e < hi; ++e) s_off[e] -= s_counts[e];
  __syncwarp();
  if (cta0) {
    for (int32_t e = lane; e < E; e += 32) {
      a.g_counts[e] = s_counts[e];
      a.g_offsets[e] = s_off[e];
    }
    if (lane == 0) a.g_offsets[E] = s_off[E];
  }
}

// External routing: the experts with 0 < count <= max_rows, in expert order,
// their counts and packed-row offsets as the routing kernel wrote them.
__device__ __forceinline__ void decode_select(const DecodeArgs& a, int lane, int32_t* s_counts, int32_t* s_off,
                                              int32_t* s_act, int32_t* misc) {
  const int32_t E = a.E;
  const int32_t per = (E + 31) / 32;
  const int32_t lo = min(E, lane * per), hi = min(E, lo + per);
  int32_t nact = 0, cmax = 0;
  for (int32_t e = lo; e < hi; ++e) {
    const int32_t c = a.g_counts[e];
    s_counts[e] = c;
    s_off[e] = a.g_offsets[e];
    const bool sel = c > 0 && c <= a.max_rows;
    nact += sel;
    if (sel) cmax = max(cmax, c);
  }
  int32_t iact = nact;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t va = __shfl_up_sync(0xffffffffu, iact, d);
    if (lane >= d) iact += va;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, d));
  int32_t ai = iact - nact;
  for (int32_t e = lo; e < hi; ++e) {
    const int32_t c = s_counts[e];
    if (c > 0 && c <= a.max_rows) s_act[ai++] = e;
  }
  if (lane == 31) {
    misc[1] = iact;
    misc[2] = cmax;
  }
}

// Grid barrier on one 64-bit arrival counter that only grows: every launch
// runs gridDim.x CTAs and each barrier takes one arrival per CTA, so a
// barrier ends when the count reaches the next multiple of gridDim.x after
// the arrival.  The arrival is acquire-release (this CTA's stores, ordered
// before by the CTA barrier, travel with it) and the polls are acquire loads.
// Nothing needs resetting when the launch ends, so the kernel finishes
// without a final round of atomics.
__device__ __forceinline__ void decode_grid_barrier(const DecodeArgs& a, int tid, int nthreads) {
  all_warps_sync(nthreads);
  if (tid == 0) {
    uint64_t* count = reinterpret_cast<uint64_t*>(a.grid_bar);
    const uint64_t G = gridDim.x;
    const uint64_t old = atom_add_acq_rel_gpu_u64(count, 1);
    const uint64_t target = (old / G + 1) * G;
    if (old + 1 != target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu_u64(count) < target) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.err, kFlagTimeout);
          break;
        }
      }
    }
  }
  all_warps_sync(nthreads);
}

// The segment in `cur` is finished: if the warp holds only part of the
// pair's k range, park its partial tiles and let the last of the pair's warps
// sum all parts in warp order; then apply alpha and store both row tiles, and
// for each finished down tile run the combine of its 16 columns if it was the
// last tile of them (batches of at most kDecLateCombine tokens; larger ones
// combine after a second grid barrier).
__device__ __forceinline__ void decode_epilogue(const DecodeCtx& cx, const Cur& cur, float (&v)[8], int lane,
                                                float4* partial, int32_t* pcount, const int32_t* s_inv,
                                                int32_t n_act, const float* rowscale) {
  const DecodeArgs& a = cx.a;
  const int32_t up = cur.ph == 0;
  const bool pair = cx.two(cur);
  if (cx.split) {
    const int32_t KT = up ? cx.KTu : cx.KTd;
    const int32_t ra = up ? cx.ura : cx.dra;
    const int32_t first_item = ra / KT;
    const int32_t seg_lo = cur.i == first_item ? ra - cur.i * KT : 0;
    if (seg_lo != 0 || cur.kt_end != KT) {
      const uint32_t TT = (uint32_t)(up ? cx.n_up : cx.n_dn) * (uint32_t)KT;  // below 2^32 with x16
      const uint32_t Wp = (uint32_t)(up ? cx.Wu : cx.Wd);
      const int32_t side = cur.i == first_item ? 0 : 1;
      float4* slot = partial + ((cx.warp * 2 + side) * 32 + lane) * 2;
      slot[0] = make_float4(v[0], v[1], v[2], v[3]);
      slot[1] = make_float4(v[4], v[5], v[6], v[7]);
      __threadfence_block();  // the readers are warps of this CTA (shared or L1-coherent global memory)
      __syncwarp();
      // warps holding tile rows i*KT .. (i+1)*KT-1 of this phase
      const int32_t wf = (int32_t)((((uint32_t)cur.i * KT + 1) * Wp - 1) / TT);
      const int32_t wl = (int32_t)((((uint32_t)(cur.i + 1) * KT) * Wp - 1) / TT);
      int32_t last = 0;
      if (lane == 0) {
        last = atomicAdd(&pcount[wf], 1) == wl - wf;
        if (last) pcount[wf] = 0;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) return;
      __threadfence_block();
      float4 rA = make_float4(0.f, 0.f, 0.f, 0.f), rB = rA;
      for (int32_t w2 = wf; w2 <= wl; ++w2) {
        const int32_t fi = (int32_t)((TT * (uint32_t)w2) / Wp) / KT;
        const float4* u = partial + ((w2 * 2 + (cur.i == fi ? 0 : 1)) * 32 + lane) * 2;
        rA.x += u[0].x; rA.y += u[0].y; rA.z += u[0].z; rA.w += u[0].w;
        rB.x += u[1].x; rB.y += u[1].y; rB.z += u[1].z; rB.w += u[1].w;
      }
      v[0] = rA.x; v[1] = rA.y; v[2] = rA.z; v[3] = rA.w;
      v[4] = rB.x; v[5] = rB.y; v[6] = rB.z; v[7] = rB.w;
    }
  }
  const int g = lane >> 2, t = lane & 3;
  const int32_t nt = min(kDecPassTok, cur.cnt - cur.tok0);
  // bf16 path: the weights were taken times 2^-8 (alpha carries 2^8); f16
  // path (rowscale): exact weights, each token column's rows times 2^-s
  const float wfix = rowscale ? 1.0f : 256.0f;
  if (rowscale) {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] *= rowscale[cur.srow + min(2 * t + (q & 1), nt - 1)];
  }
  const float alpha = (up ? a.up_g : a.dn_g)[cur.e] * wfix;
  if (up && a.gated) {
    // the pair is (gate tile, up tile) of the same 16 intermediate rows
    const float ag = a.gate_g[cur.e] * wfix;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int32_t col = 2 * t + (q & 1);
      const int32_t row = (cur.rt >> 1) * 16 + g + 8 * (q >> 1);
      if (col < nt) {
        const size_t pr = (size_t)(cur.off + cur.tok0 + col);
        const float gv = v[q] * ag;
        a.Ap[pr * a.I + row] = f2bf_rn(gv / (1.0f + expf(-gv)) * (v[4 + q] * alpha));
      }
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int32_t col = 2 * t + (q & 1);
    const int32_t row = (cur.rt + (q >> 2)) * 16 + g + 8 * ((q >> 1) & 1);
    if (col < nt && (q < 4 || pair)) {
      const size_t pr = (size_t)(cur.off + cur.tok0 + col);
      const float h = v[q] * alpha;
      if (up) {
        const float rl = h > 0.0f ? h : 0.0f;
        a.Ap[pr * a.I + row] = f2bf_rn(rl * rl);
      } else {
        a.Yp[pr * a.H + row] = h;
      }
    }
  }
  if (up || a.ext || a.n > kDecLateCombine || cur.tok0 + kDecPassTok < cur.cnt) return;
  // down tiles complete: count each against its 16 columns.  The warp
  // barrier orders every lane's row stores before lane 0's acquire-release
  // count, which publishes them (cumulatively) to the last counter of the
  // block; its acquire, and the warp barrier after it, make every tile's
  // rows visible to the lanes that combine them.
  __syncwarp();
  for (int h = 0; h < (pair ? 2 : 1); ++h) {
    const int32_t rt = cur.rt + h;
    int32_t last = 0;
    if (lane == 0) {
      last = atom_add_acq_rel_gpu(&a.col_done[rt], 1) == n_act - 1;
      if (last) a.col_done[rt] = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __syncwarp();
    const int32_t c = rt * 16 + (lane & 15);
    for (int32_t tk = lane >> 4; tk < a.n; tk += 2) {
      const size_t o = (size_t)tk * a.H + c;
      float acc = __uint_as_float((uint32_t)a.dst[o] << 16);
      for (int32_t j = 0; j < a.k; ++j) {
        const int32_t r = s_inv[tk * a.k + j];
        if (r >= 0) acc = __fmaf_rn(a.tw[tk * a.k + j], ld_cg_f32(a.Yp + (size_t)r * a.H + c), acc);
      }
      a.dst_out[o] = f2bf_rn(acc);
    }
  }
}

// dst[t][c] = bf16(dst[t][c] + sum_j w[t][j] * Yp[inv[t][j]][c]) for one
// element, j in order; the k row loads are issued before the FMA chain.
__device__ __forceinline__ void combine_one(const DecodeArgs& a, const int32_t* s_inv, int32_t tk, int32_t c) {
  const size_t o = (size_t)tk * a.H + c;
  float acc = __uint_as_float((uint32_t)a.dst[o] << 16);
  for (int32_t j0 = 0; j0 < a.k; j0 += 8) {
    int32_t r[8];
    float y[8], w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int32_t j = j0 + q;
      r[q] = j < a.k ? s_inv[tk * a.k + j] : -1;
      y[q] = r[q] >= 0 ? ld_cg_f32(a.Yp + (size_t)r[q] * a.H + c) : 0.f;
      w[q] = r[q] >= 0 ? a.tw[tk * a.k + j] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (r[q] >= 0) acc = __fmaf_rn(w[q], y[q], acc);
  }
  a.dst_out[o] = f2bf_rn(acc);
}

// bf16 pair w times `down` (a power of two) as an f16 pair.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float down) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * down, __uint_as_float(w & 0xFFFF0000u) * down);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t w, uint32_t m) {
  return max(m, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu));
}

// All threads of the CTA: wait for phase ph's staged bf16 rows, then rewrite
// each in place as f16 values times 2^-s, with s per row putting the row's
// largest magnitude in [2^14, 2^15) (s clamped to [-126, 126]), and keep 2^s
// for the epilogue.  A bf16 value is then an f16 number exactly unless its
// scaled magnitude is below 2^-14 -- 2^28 under the row's largest -- where the
// f16 subnormal spacing 2^-24 rounds it.  The CTA barrier at the end orders
// the rewritten rows before any fragment load.  Returns false if the wait
// ran out (the rows are then left as they are).
__device__ bool stage_to_f16(const DecodeCtx& cx, int32_t ph, uint64_t* bar, float* rowscale, int warp, int lane,
                             int nwarps, int nthreads) {
  bool ok = mbar_wait_sleep(bar, (uint32_t)ph, cx.a.err);
  ok = !__any_sync(0xffffffffu, !ok);
  const int32_t* sb = ph ? cx.sbd : cx.sbu;
  const int32_t span = ph ? cx.span_d : cx.span_u;
  const int32_t rows = span > 0 ? sb[span] : 0;
  const int32_t n8 = (ph ? cx.a.I : cx.a.H) / 8;
  const uint32_t RS = ph ? cx.RSd : cx.RSu;
  for (int32_t r = warp; ok && r < rows; r += nwarps) {
    uint4* row = reinterpret_cast<uint4*>(cx.stage + (size_t)r * RS);
    uint32_t mx = 0;
    for (int32_t i = lane; i < n8; i += 32) {
      const uint4 v = row[i];
      mx = bf16x2_absmax(v.x, bf16x2_absmax(v.y, bf16x2_absmax(v.z, bf16x2_absmax(v.w, mx))));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    // floor(log2) of the largest magnitude: the bf16 exponent, or for a
    // subnormal (value m * 2^-133) the top bit of its mantissa
    const int32_t lg = (mx >> 7) ? (int32_t)(mx >> 7) - 127 : (31 - __clz((int)mx)) - 133;
    const int32_t s = mx ? min(126, max(-126, lg - 14)) : 0;
    const float down = __uint_as_float((uint32_t)(127 - s) << 23);
    if (lane == 0) rowscale[r] = __uint_as_float((uint32_t)(127 + s) << 23);
    for (int32_t i = lane; i < n8; i += 32) {
      const uint4 v = row[i];
      row[i] = make_uint4(bf16x2_to_f16x2_scaled(v.x, down), bf16x2_to_f16x2_scaled(v.y, down),
                          bf16x2_to_f16x2_scaled(v.z, down), bf16x2_to_f16x2_scaled(v.w, down));
    }
  }
  all_warps_sync(nthreads);
  return ok;
}

// One warp from its ring fill through the grid barrier to the drain of its
// copies.  STAGED: the activation fragments come from the CTA-wide stage,
// otherwise from each chunk's own activation copies (compiled separately so
// that neither loop carries the other's addressing).
template <bool STAGED>
__device__ __forceinline__ void decode_stream(const DecodeArgs& a, const DecodeCtx& cx, uint8_t* ring,
                                              uint32_t slot_bytes, int32_t P, uint64_t* wbar, Cur* wdesc,
                                              uint64_t* stage_bar, const uint32_t* lut, const uint32_t* lut16,
                                              float* rowscale, float4* partial, int32_t* pcount,
                                              const int32_t* s_inv, int32_t n_act, int tid, int nthreads) {
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t wbytes = cx.wbytes;
  const uint64_t pol = policy_evict_first();

  // Chunk q of this warp's sequence lives in slot q % P.  Its weights are
  // requested P chunks ahead; its activations too, except down chunks issued
  // before the grid barrier, whose activations follow right after it.
  Cur ci;
  cx.template enter_phase<STAGED>(ci, 0);
  int32_t issued = 0, acts_issued = 0;
  bool crossed = false, dead = false;
  auto issue = [&](int32_t s) {
    uint8_t* sp = ring + (size_t)s * slot_bytes;
    if (lane == 0) {
      wdesc[s] = ci;
      cx.template issue_weights<STAGED>(ci, sp, &wbar[s], pol);
    }
    if (ci.ph == 0 || crossed) {
      cx.template issue_acts<STAGED>(ci, lane, sp, &wbar[s]);
      ++acts_issued;
    }
    cx.template advance<STAGED>(ci);
    ++issued;
  };
  // The up phase's staged activation rows go first, then the rings fill in
  // rounds -- every warp's first chunk, then every warp's second, ... -- so
  // that the copies needed first lead the SM's copy queue.
  int32_t stage_issued = 0;
  if (STAGED && warp == 0) {
    cx.issue_stage(0, lane, stage_bar);
    stage_issued = 1;
  }
  for (int32_t s = 0; s < P; ++s) {
    if (ci.ph < 2) issue(s);
    all_warps_sync(nthreads);
  }
  // staged rows become scaled f16 rows once they land (every warp helps)
  if (STAGED && !stage_to_f16(cx, 0, stage_bar, rowscale, warp, lane, nthreads >> 5, nthreads)) dead = true;

  int32_t consumed = 0, slot = 0;
  uint32_t phase = 0;
  float accA[4] = {0.f, 0.f, 0.f, 0.f}, accA2[4] = {0.f, 0.f, 0.f, 0.f};
  float accB[4] = {0.f, 0.f, 0.f, 0.f}, accB2[4] = {0.f, 0.f, 0.f, 0.f};
  while (!dead && consumed < issued) {
    const Cur cur = wdesc[slot];
    if (cur.ph == 1 && !crossed) {
      // every up tile of every CTA is stored before any down tile reads Ap
      decode_grid_barrier(a, tid, nthreads);
      crossed = true;
      if (STAGED) {
        if (warp == 0) {
          cx.issue_stage(1, lane, stage_bar);
          stage_issued = 2;
        }
        if (!stage_to_f16(cx, 1, stage_bar, rowscale, warp, lane, nthreads >> 5, nthreads)) {
          dead = true;
          break;
        }
      }
      for (int32_t q = acts_issued; q < issued; ++q) {
        const int32_t s = q % P;
        cx.template issue_acts<STAGED>(wdesc[s], lane, ring + (size_t)s * slot_bytes, &wbar[s]);
      }
      acts_issued = issued;
    }
    const bool ok = mbar_wait_sleep(&wbar[slot], phase, a.err);
    if (__any_sync(0xffffffffu, !ok)) {
      dead = true;
      break;
    }
    if (consumed == 0 && lane == 0) {
      // once the first chunk has landed, ask L2 for the chunks past the ring
      Cur cp = ci;
      for (int q = 0; q < kDecL2Ahead && cp.ph < 2; ++q) {
        const uint8_t* src = cx.template chunk_src<STAGED>(cp);
        prefetch_l2_bulk(src, (uint32_t)cx.kts(cp) * kTileBytes);
        if (cx.two(cp))
          prefetch_l2_bulk(src + (size_t)(cp.ph ? cx.KTd : cx.KTu) * kTileBytes, (uint32_t)cx.kts(cp) * kTileBytes);
        cx.template advance<STAGED>(cp);
      }
    }
    const uint8_t* sp = ring + (size_t)slot * slot_bytes;
    const int32_t nt = min(kDecPassTok, cur.cnt - cur.tok0);
    const int32_t col = min(lane >> 2, nt - 1);
    const uint8_t* act =
        STAGED ? cx.stage + (size_t)(cur.srow + col) * (cur.ph ? cx.RSd : cx.RSu) + cur.kt * 128 + (lane & 3) * 32
               : sp + wbytes + col * kDecActRow + (lane & 3) * 32;
    if (STAGED)
      chunk_mma16(sp, act, cx.kts(cur), cx.two(cur), lane, lut16, accA, accA2, accB, accB2);
    else
      chunk_mma(sp, act, cx.kts(cur), cx.two(cur), lane, lut, accA, accA2, accB, accB2);
    ++consumed;
    __syncwarp();
    if (ci.ph < 2) {
      if (lane == 0) fence_proxy_async_smem();
      issue(slot);
      __syncwarp();
    }
    if (++slot == P) {
      slot = 0;
      phase ^= 1u;
    }
    if (cur.kt + kDecCK >= cur.kt_end) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q] = accA[q] + accA2[q];
        v[4 + q] = accB[q] + accB2[q];
        accA[q] = accA2[q] = accB[q] = accB2[q] = 0.f;
      }
      decode_epilogue(cx, cur, v, lane, partial, pcount, s_inv, n_act, STAGED ? rowscale : nullptr);
    }
  }
  if (!crossed) {
    decode_grid_barrier(a, tid, nthreads);
    if (STAGED) {
      if (warp == 0) {
        cx.issue_stage(1, lane, stage_bar);
        stage_issued = 2;
      }
      if (!stage_to_f16(cx, 1, stage_bar, rowscale, warp, lane, nthreads >> 5, nthreads)) dead = true;
    }
  }
  if (stage_issued > 0) {
    // (warp 0) the stage copies it issued land before the CTA can exit; the
    // last phase issued completes after the earlier one
    mbar_wait_sleep(stage_bar, (uint32_t)(stage_issued - 1), a.err);
  }
  if (dead) {
    // let this warp's copies still in flight land before the CTA exits; the
    // chunks whose activations were never requested get them now (in-bounds
    // reads of whatever the rows hold) so that their barriers can complete
    for (int32_t q = acts_issued; q < issued; ++q) {
      const int32_t s = q % P;
      cx.template issue_acts<STAGED>(wdesc[s], lane, ring + (size_t)s * slot_bytes, &wbar[s]);
    }
    for (int32_t q = consumed; q < issued; ++q) mbar_wait_sleep(&wbar[q % P], (uint32_t)((q / P) & 1), a.err);
  }
}

// CAN_STAGE = false compiles the per-chunk activation path alone: a batch of
// one token has one token per expert, where staging never applies, and that
// loop then keeps the registers and code layout it has on its own.
template <bool CAN_STAGE>
__global__ void __launch_bounds__(kDecMaxWarps * 32, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const DecLayout& L = a.L;
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.scale_lut);
  uint32_t* lut16 = reinterpret_cast<uint32_t*>(smem + L.scale_lut16);
  float* rowscale = reinterpret_cast<float*>(smem + L.rowexp);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + L.ids);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem + L.perm);
  int32_t* s_inv = reinterpret_cast<int32_t*>(smem + L.inv);
  int32_t* s_counts = reinterpret_cast<int32_t*>(smem + L.counts);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + L.offsets);
  int32_t* s_act = reinterpret_cast<int32_t*>(smem + L.act);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.misc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* stage_bar = bars + kDecMaxSlots * kDecMaxWarps;
  int32_t* s_sbase = reinterpret_cast<int32_t*>(smem + L.sbase);
  float4* partial = CAN_STAGE ? a.partial + (size_t)blockIdx.x * kDecPartialPerCta
                              : reinterpret_cast<float4*>(smem + L.partial);
  int32_t* pcount = reinterpret_cast<int32_t*>(smem + L.pcount);
  Cur* descs = reinterpret_cast<Cur*>(smem + L.desc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, W = nthreads >> 5;
  const int32_t R = a.n * a.k, E = a.E;

  if (!a.ext) {
    for (int32_t i = tid; i < R; i += nthreads) s_ids[i] = a.ids[i];
    for (int32_t i = tid; i < E; i += nthreads) s_counts[i] = 0;
  }
  if (!a.ext && warp == 1 && lane == 0) {
    // While the routing is worked out, ask L2 for the up weights of the picked
    // experts (a slice per CTA of their concatenation in pair order), when
    // they fit well inside L2: the ring's first requests then find them there.
    // (32-bit arithmetic once the total is known to be below 48 MB: this
    // thread's divisions would otherwise hold up the CTA's first barrier)
    const uint32_t per = (uint32_t)((a.gated ? 2 * a.I : a.I) / 16) * (uint32_t)(a.H / 64) * kTileBytes;
    if ((int64_t)R * per <= kDecEarlyL2Bytes) {
      const uint32_t total = (uint32_t)R * per;
      const uint32_t share = ((total + gridDim.x - 1) / gridDim.x + 15u) & ~15u;
      uint32_t lo = blockIdx.x * share;
      const uint32_t hi = min(total, lo + share);
      // (batches of several tokens mostly stream the f16 path's tiles)
      const uint8_t* tiles = CAN_STAGE ? a.up_tiles16 : a.up_tiles;
      while (lo < hi) {
        const uint32_t j = lo / per, off = lo - j * per;
        const uint32_t len = min(min(per - off, hi - lo), 65536u);
        const int32_t e = __ldg(a.ids + j);
        if (e >= 0 && e < E && len >= 16) prefetch_l2_bulk(tiles + (size_t)e * per + off, len & ~15u);
        lo += len;
      }
    }
  }
  for (int i = tid; i < 256; i += nthreads) lut[i] = scale_bf16_2p118((uint32_t)i) * 0x10001u;
  if (CAN_STAGE)
    for (int i = tid; i < 256; i += nthreads) lut16[i] = scale_f16x2((uint32_t)i);
  for (int i = tid; i < kDecMaxWarps; i += nthreads) pcount[i] = 0;
  if (lane == 0) {
    // one arrival: lane 0's expect_tx covering the weight and activation copies
    for (int q = 0; q < kDecMaxSlots; ++q) mbar_init(&bars[warp * kDecMaxSlots + q], 1);
    if (warp == 0) mbar_init(stage_bar, 1);  // one arrival per phase: warp 0 lane 0's expect_tx
    fence_mbar_init();
  }
  __syncthreads();
  if (a.ext) {
    if (warp == 0) decode_select(a, lane, s_counts, s_off, s_act, misc);
  } else {
    bool bad = false;
    for (int32_t p = tid; p < R; p += nthreads) {
      const int32_t e = s_ids[p];
      if (e >= 0 && e < E) atomicAdd(&s_counts[e], 1);
      else bad = true;
    }
    if (bad && blockIdx.x == 0) atomicOr(a.err, kFlagBadRouting);
    __syncthreads();
    if (warp == 0) decode_route(a, lane, s_ids, s_tok, s_inv, s_counts, s_off, s_act, misc);
  }
  if (CAN_STAGE && warp == 0) decode_stage_plan(a, lane, s_counts, s_act, misc, s_sbase);
  __syncthreads();

  const int32_t n_act = misc[1], cmax = misc[2];
  // slot size follows the widest token pass; keep at least two slots per warp
  const uint32_t nt_cap = (uint32_t)max(1, min(kDecPassTok, cmax));
  // two row tiles per work item once an expert has several tokens (their
  // activation fragments are then loaded once for both); single tiles keep
  // the chunks small where the layer is all latency.  A gated up projection
  // always takes its gate and up tiles together.
  const DecItems it = dec_items(a, n_act, cmax);
  const int32_t pd = it.pd, pu = it.pu;
  const uint32_t wbytes = pu ? kDecSlotBytes : kDecCK * kTileBytes;
  // Staged rows replace the activation part of every slot; stage only if
  // that leaves at least as many streaming warps as per-chunk copies would.
  const uint32_t region = L.total - L.ring;
  const uint32_t copy_slot = wbytes + nt_cap * kDecActRow;
  const int32_t W_copy = max(1, min(W, (int32_t)(region / (2u * copy_slot))));
  const bool plan_ok = CAN_STAGE && misc[3] != 0;
  const uint32_t planned = plan_ok ? (uint32_t)misc[4] : region;
  const int32_t W_stage = planned < region ? max(1, min(W, (int32_t)((region - planned) / (2u * wbytes)))) : 0;
  const bool staged = plan_ok && W_stage >= W_copy;
  const uint32_t stage_bytes = staged ? planned : 0u;
  const uint32_t slot_bytes = staged ? wbytes : copy_slot;
  const uint32_t ring_bytes = region - stage_bytes;
  const int32_t Weff = staged ? W_stage : W_copy;
  const int32_t P = min(kDecMaxSlots, (int32_t)(ring_bytes / ((uint32_t)Weff * slot_bytes)));

  DecodeCtx cx(a);
  cx.s_tok = s_tok; cx.s_counts = s_counts; cx.s_off = s_off; cx.s_act = s_act;
  cx.warp = warp; cx.W = Weff;
  cx.KTu = a.H / 64; cx.KTd = a.I / 64; cx.NTu = (a.gated ? 2 * a.I : a.I) / 16; cx.NTd = a.H / 16;
  cx.pu = pu; cx.pd = pd; cx.wbytes = wbytes;
  cx.NPu = it.NPu; cx.NPd = it.NPd;
  cx.staged = staged;
  cx.stage = smem + L.total - stage_bytes;
  cx.RSu = 2u * (uint32_t)a.H + 16u;
  cx.RSd = 2u * (uint32_t)a.I + 16u;
  cx.sbu = s_sbase;
  cx.sbd = s_sbase + (kDecMaxSpan + 1);
  cx.elo_u = misc[5]; cx.span_u = misc[6]; cx.elo_d = misc[7]; cx.span_d = misc[8];
  {
    cx.u_lo = it.u_lo;
    cx.d_lo = it.d_lo;
    cx.n_up = it.n_up;
    cx.n_dn = it.n_dn;
    cx.split = cmax <= kDecPassTok;
    // k-tiles per phase and CTA: at most 262144 items (E <= 1024, 256 per
    // expert) x 64 k-tiles, times at most 16 warps, stays below 2^32
    const uint32_t TTu = (uint32_t)cx.n_up * (uint32_t)cx.KTu, TTd = (uint32_t)cx.n_dn * (uint32_t)cx.KTd;
    cx.Wu = (int32_t)(TTu < (uint32_t)Weff ? TTu : (uint32_t)Weff);
    cx.Wd = (int32_t)(TTd < (uint32_t)Weff ? TTd : (uint32_t)Weff);
    cx.ura = warp < cx.Wu ? (int32_t)(TTu * (uint32_t)warp / (uint32_t)cx.Wu) : 0;
    cx.urb = warp < cx.Wu ? (int32_t)(TTu * (uint32_t)(warp + 1) / (uint32_t)cx.Wu) : 0;
    cx.dra = warp < cx.Wd ? (int32_t)(TTd * (uint32_t)warp / (uint32_t)cx.Wd) : 0;
    cx.drb = warp < cx.Wd ? (int32_t)(TTd * (uint32_t)(warp + 1) / (uint32_t)cx.Wd) : 0;
  }
  uint8_t* ring = smem + L.ring + (size_t)min(warp, Weff - 1) * P * slot_bytes;
  uint64_t* wbar = bars + warp * kDecMaxSlots;
  Cur* wdesc = descs + warp * kDecMaxSlots;
  if (CAN_STAGE && staged)
    decode_stream<true>(a, cx, ring, slot_bytes, P, wbar, wdesc, stage_bar, lut, lut16, rowscale, partial, pcount,
                        s_inv, n_act, tid, nthreads);
  else
    decode_stream<false>(a, cx, ring, slot_bytes, P, wbar, wdesc, stage_bar, lut, lut16, rowscale, partial, pcount,
                         s_inv, n_act, tid, nthreads);
  if (!a.ext && a.n > kDecLateCombine) {
    // every down row of every CTA is stored: combine, one element per thread
    decode_grid_barrier(a, tid, nthreads);
    const int64_t total = (int64_t)a.n * a.H, stride = (int64_t)gridDim.x * nthreads;
    for (int64_t idx = (int64_t)blockIdx.x * nthreads + tid; idx < total; idx += stride)
      combine_one(a, s_inv, (int32_t)(idx / a.H), (int32_t)(idx % a.H));
  }
}

DecLayout decode_layout(int32_t E, int32_t R, bool can_stage) {
  return dec_layout(E, R, 227 * 1024 - 1024, !can_stage);
}

cudaError_t launch_decode(const DecodeArgs& args, int num_sms, cudaStream_t s) {
  static std::atomic<bool> attr_set[2][kMaxDevices];
  const bool can_stage = decode_can_stage(args.n, args.ext);
  auto kernel = can_stage ? decode_kernel<true> : decode_kernel<false>;
  cudaError_t e = raise_smem_limit(kernel, 227 * 1024, attr_set[can_stage ? 1 : 0]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms);
  cfg.blockDim = dim3(args.L.warps * 32);
  cfg.dynamicSmemBytes = args.L.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace moe
