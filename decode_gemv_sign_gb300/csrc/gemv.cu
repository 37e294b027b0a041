// Fused decode-GEMV and the plain BF16 GEMV it is compared against.
//
//   y[b, r] = sum_k x[b, k] * W[r, k],   b < B <= 16,  r < N
//
// Method: forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un
// 25%", section "Qué queda por demostrar": codes rebuilt in registers inside
// the GEMV, with the sparse escape correction applied in the same kernel (the
// pages' own prototype left it unfused).  wavect page "Compresión de pesos LLM
// sin pérdida vs 8-bit GGUF", section "¿Qué significa “sin pérdida” para los
// pesos de un LLM?": exact BF16 rebuilt in registers and used at once.
//
// Two kernels compute it: the FMA kernel below (small batches of the
// encoded sources) and the tensor-core kernel further down (larger batches,
// and the plain GEMV at every batch); mma_min_batch() holds the measured
// crossover per source.  Both take their units from the same kind of global
// counter and give results independent of scheduling.
//
// FMA kernel.  A unit of work is a set of R consecutive rows of one
// tensor; a launch covers the units of every tensor in the batch.  The grid is
// persistent (as many CTAs as fit on the GPU at once) and every warp grabs
// units from a global counter, one at a time, so the GPU drains evenly even
// when the tensors differ in shape.  Inside a unit the warp walks the rows in
// 1024-element chunks (lane mapping below), keeps the next chunk's loads in
// flight while it computes the current one (register double buffering),
// loads the streams with coalesced loads that bypass L1, rebuilds BF16 pairs
// with prmt lookups and accumulates in fp32 (mixed-precision or packed
// fp32x2 FMAs, see below).  x is read through L1, where it stays (every warp
// of the SM reads the same x).
//
// Escapes.  An escaped weight decodes to the placeholder (symbol 0, so
// |w| < 2^-125).  Each lane adds x * (w_true - w_placeholder) for a share of
// the unit's escapes, found in O(1) through the row index; the first 32
// positions and values are requested when the unit starts, so those loads
// overlap its chunks, and the corrections are added when it ends.  Lanes are
// combined with a fixed butterfly: results do not depend on which warp ran
// which unit.
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "wcomp_impl.cuh"

namespace wc {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlots = 1024;  // work-counter slots per device (one per launch, round robin)

enum Src { kBytesplit = WCOMP_BYTESPLIT, kK15 = WCOMP_K15, kPlain = 2 };

// Build-time choices: the staged (TMA) kernel or the register double-buffered
// kernel, and the proxy fence before a stage is refilled.
#ifndef WCOMP_GEMV_TMA
#define WCOMP_GEMV_TMA 0
#endif
#ifndef WCOMP_GEMV_MODE1
#define WCOMP_GEMV_MODE1 1
#endif

#ifndef WCOMP_GEMV_MINB1
#define WCOMP_GEMV_MINB1 4
#endif
#ifndef WCOMP_GEMV_MINB1_K15
#define WCOMP_GEMV_MINB1_K15 3
#endif
#ifndef WCOMP_GEMV_PROXY_FENCE
#define WCOMP_GEMV_PROXY_FENCE 1
#endif

// FMA forms.  MODE 0 widens weights and x to fp32 and issues packed fp32x2
// FMAs (x is widened once per unit of R rows).  MODE 1 feeds the BF16 halves
// of the pair words straight into mixed-precision FMAs (bf16 x bf16 + fp32);
// the product of two BF16 values is exact in fp32, so both forms round the
// same sums.  MODE 1 saves the widening work and wins for small batches.
#ifndef WCOMP_GEMV_MIXED_MAX_B
#define WCOMP_GEMV_MIXED_MAX_B 4
#endif

__device__ __forceinline__ void fma_wide(float2& acc, uint32_t w_pair, float x0, float x1) {
  acc = __ffma2_rn(make_float2(bf16_lo(w_pair), bf16_hi(w_pair)), make_float2(x0, x1), acc);
}

__device__ __forceinline__ void fma_mixed(float2& acc, uint32_t w_pair, uint32_t x_pair) {
  unsigned short w0, w1, x0, x1;
  asm("mov.b32 {%0, %1}, %2;" : "=h"(w0), "=h"(w1) : "r"(w_pair));
  asm("mov.b32 {%0, %1}, %2;" : "=h"(x0), "=h"(x1) : "r"(x_pair));
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc.x) : "h"(w0), "h"(x0));
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc.y) : "h"(w1), "h"(x1));
}

__device__ __forceinline__ uint4 ld_x_v4(const uint16_t* p) {
  uint4 v;
  asm("ld.global.nc.L1::evict_last.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Loads at a base address plus a compile-time byte offset: the offset goes
// into the instruction, so the slices of a chunk share one address register.
template <int OFF>
__device__ __forceinline__ uint32_t ld_stream_u32_at(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1+%2];" : "=r"(v) : "l"(p), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 ld_stream_v2_at(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "l"(p), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 ld_stream_v4_at(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 ld_x_v4_at(const uint16_t* p) {
  uint4 v;
  asm("ld.global.nc.L1::evict_last.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "n"(OFF));
  return v;
}

// Find the tensor that owns global unit `u`, searching from tensor `start`
// (a warp's units only increase, so its previous owner is a lower bound).
__device__ __forceinline__ int owner(const uint32_t* prefix, int count, uint32_t u, int start = 0) {
  int i = start;
  while (i + 1 < count && prefix[i + 1] <= u) ++i;
  return i;
}

// ---------------------------------------------------------------------------
// Lane mapping.  A row is walked in chunks of 1024 elements.  Inside a chunk,
// lane l owns the four 8-element slices starting at 256 i + 8 l (i = 0..3):
// for every slice the 32 lanes cover 256 consecutive elements, so each load
// of codes (4 bytes), raw bytes (8), mantissa-plane words, plain BF16 (16)
// and x (16) is one contiguous, fully coalesced request per warp.
// ---------------------------------------------------------------------------
constexpr int kChunk = 1024;
constexpr int kSlice = 256;

// One row's share of a chunk for one lane.
//   byte-split: v[i] code word of slice i, v[4+2i], v[5+2i] its raw bytes
//   K15:        v[i] code word, v[4+i] plane A word, v[8+i] plane B word,
//               v[12+i] plane C word (shared by the 4 lanes of a 32-element group)
//   plain:      v[4i .. 4i+3] the slice's 8 BF16 values
struct ChunkBuf {
  uint32_t v[16];
};

// Stream base pointers of one tensor, held in registers for a unit.
struct Streams {
  const uint8_t *codes, *raw, *pa, *pb, *pc;
};

// Slice I of one row's chunk; `q` holds the lane's stream addresses for
// slice 0 (chunk_ptrs), the slice offsets are immediates.
struct ChunkPtrs {
  const uint8_t *c, *r, *a, *b, *cc;
};

// e_base is the chunk's first element; it is a multiple of 32 (K % 32 == 0).
template <int SRC>
__device__ __forceinline__ ChunkPtrs chunk_ptrs(const Streams& d, uint64_t e_base, int lane) {
  ChunkPtrs q{};
  if (SRC == kBytesplit) {
    q.c = d.codes + (e_base >> 1) + 4 * lane;
    q.r = d.raw + e_base + 8 * lane;
  } else if (SRC == kK15) {
    // group g = e >> 5 of element e = e_base + 256 i + 8 lane; the lane reads
    // quads 2 (lane & 3), +1: plane A word 16 g + 4 (lane & 3), plane B word
    // 8 g + 4 ((lane >> 1) & 1), plane C word 4 g
    q.c = d.codes + (e_base >> 1) + 4 * lane;
    q.a = d.pa + (e_base >> 1) + 4 * lane;
    q.b = d.pb + (e_base >> 2) + 8 * (lane >> 2) + 4 * ((lane >> 1) & 1);
    q.cc = d.pc + (e_base >> 3) + 4 * (lane >> 2);
  } else {
    q.r = d.raw + 2 * e_base + 16 * lane;
  }
  return q;
}

template <int SRC, int I>
__device__ __forceinline__ void load_slice(const ChunkPtrs& q, ChunkBuf& b) {
  if (SRC == kBytesplit) {
    b.v[I] = ld_stream_u32_at<128 * I>(q.c);
    const uint2 r = ld_stream_v2_at<256 * I>(q.r);
    b.v[4 + 2 * I] = r.x;
    b.v[5 + 2 * I] = r.y;
  } else if (SRC == kK15) {
    b.v[I] = ld_stream_u32_at<128 * I>(q.c);
    b.v[4 + I] = ld_stream_u32_at<128 * I>(q.a);
    b.v[8 + I] = ld_stream_u32_at<64 * I>(q.b);
    b.v[12 + I] = ld_stream_u32_at<32 * I>(q.cc);
  } else {
    const uint4 w = ld_stream_v4_at<512 * I>(q.r);
    b.v[4 * I + 0] = w.x; b.v[4 * I + 1] = w.y; b.v[4 * I + 2] = w.z; b.v[4 * I + 3] = w.w;
  }
}

// Loads of one row's chunk in address form ADDR (see addr_mode).
template <int SRC, bool FULL, int ADDR>
__device__ __forceinline__ void load_chunk(const Streams& d, uint64_t e_base, uint32_t vmask, int lane,
                                           ChunkBuf& b) {
  if (ADDR == 2) {
    // lane l holds elements 32 l .. +31 of the chunk (one whole group); in a
    // partial chunk vmask is 0xF or 0 per lane
    if (!FULL && !vmask) return;
    const uint64_t e = e_base + 32 * uint64_t(lane);
    if (SRC == kPlain) {
      uint32_t r[8];
      ld_stream_v8(d.raw + 2 * e, r);
#pragma unroll
      for (int k = 0; k < 8; ++k) b.v[k] = r[k];
      ld_stream_v8(d.raw + 2 * e + 32, r);
#pragma unroll
      for (int k = 0; k < 8; ++k) b.v[8 + k] = r[k];
      return;
    }
    const uint4 c = ld_stream_v4(d.codes + (e >> 1));
    b.v[0] = c.x; b.v[1] = c.y; b.v[2] = c.z; b.v[3] = c.w;
    if (SRC == kBytesplit) {
      uint32_t r[8];
      ld_stream_v8(d.raw + e, r);
#pragma unroll
      for (int k = 0; k < 8; ++k) b.v[4 + k] = r[k];
    } else {
      const uint4 a = ld_stream_v4(d.pa + (e >> 1));
      b.v[4] = a.x; b.v[5] = a.y; b.v[6] = a.z; b.v[7] = a.w;
      const uint2 bb = ld_stream_v2(d.pb + (e >> 2));
      b.v[8] = bb.x; b.v[9] = bb.y;
      b.v[12] = ld_stream_u32(d.pc + (e >> 3));
    }
    return;
  }
  if (ADDR == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!FULL && !((vmask >> i) & 1)) continue;
      const uint64_t e = e_base + kSlice * i + 8 * lane;
      if (SRC == kBytesplit) {
        b.v[i] = ld_stream_u32(d.codes + (e >> 1));
        const uint2 r = ld_stream_v2(d.raw + e);
        b.v[4 + 2 * i] = r.x;
        b.v[5 + 2 * i] = r.y;
      } else if (SRC == kK15) {
        const uint64_t g = e >> 5;
        const uint32_t q2 = lane & 3;
        b.v[i] = ld_stream_u32(d.codes + (e >> 1));
        b.v[4 + i] = ld_stream_u32(d.pa + 16 * g + 4 * q2);
        b.v[8 + i] = ld_stream_u32(d.pb + 8 * g + 4 * (q2 >> 1));
        b.v[12 + i] = ld_stream_u32(d.pc + 4 * g);
      } else {
        const uint4 w = ld_stream_v4(d.raw + 2 * e);
        b.v[4 * i + 0] = w.x; b.v[4 * i + 1] = w.y; b.v[4 * i + 2] = w.z; b.v[4 * i + 3] = w.w;
      }
    }
    return;
  }
  const ChunkPtrs q = chunk_ptrs<SRC>(d, e_base, lane);
  if (FULL || (vmask & 1)) load_slice<SRC, 0>(q, b);
  if (FULL || (vmask & 2)) load_slice<SRC, 1>(q, b);
  if (FULL || (vmask & 4)) load_slice<SRC, 2>(q, b);
  if (FULL || (vmask & 8)) load_slice<SRC, 3>(q, b);
}

// BF16 pairs (elements 2q, 2q+1 of the slice in w[q]) of slice I.
template <int SRC, int I>
__device__ __forceinline__ void slice_pairs(const RegTable& t, const ChunkBuf& b, int lane, uint32_t (&w)[4]) {
  if (SRC == kPlain) {
    w[0] = b.v[4 * I + 0]; w[1] = b.v[4 * I + 1]; w[2] = b.v[4 * I + 2]; w[3] = b.v[4 * I + 3];
    return;
  }
  const uint32_t cw = b.v[I];
  const QuadMasks m = code_masks(cw);
  const uint32_t m7 = cw & 0x77777777u;
  uint32_t h0, h1, l0, l1;
  lookup8(t.hi, m7, m, h0, h1);
  if (SRC == kBytesplit) {
    l0 = b.v[4 + 2 * I];
    l1 = b.v[5 + 2 * I];
  } else {
    // quads q0 = 2 (lane & 3) and q0 + 1 of the 32-element group
    const uint32_t A = b.v[4 + I], Bw = b.v[8 + I], C = b.v[12 + I];
    const uint32_t q0 = 2 * (lane & 3), sb0 = 4 * (lane & 1);
    uint32_t e0, e1;
    lookup8(t.e0, m7, m, e0, e1);
    l0 = (A & 0x0F0F0F0Fu) | (((Bw >> sb0) << 4) & 0x30303030u) | (((C >> q0) << 6) & 0x40404040u) | e0;
    l1 = ((A >> 4) & 0x0F0F0F0Fu) | (((Bw >> (sb0 + 2)) << 4) & 0x30303030u) |
         (((C >> (q0 + 1)) << 6) & 0x40404040u) | e1;
  }
  w[0] = prmt(l0, h0, 0x5140);
  w[1] = prmt(l0, h0, 0x7362);
  w[2] = prmt(l1, h1, 0x5140);
  w[3] = prmt(l1, h1, 0x7362);
}

// K15 pairs of slice I of a lane that holds a whole 32-element group (its
// four slices are the group's four quarters, so the plane bit positions are
// compile-time constants): code word v[I], plane A word v[4 + I], plane B
// word v[8 + I / 2], plane C word v[12].
template <int I>
__device__ __forceinline__ void group_slice_pairs_k15(const RegTable& t, const ChunkBuf& b, uint32_t (&w)[4]) {
  const uint32_t cw = b.v[I];
  const QuadMasks m = code_masks(cw);
  const uint32_t m7 = cw & 0x77777777u;
  uint32_t h0, h1, e0, e1;
  lookup8(t.hi, m7, m, h0, h1);
  lookup8(t.e0, m7, m, e0, e1);
  const uint32_t A = b.v[4 + I], Bw = b.v[8 + (I >> 1)], C = b.v[12];
  constexpr int sb0 = 4 * (I & 1), q0 = 2 * I;
  const uint32_t l0 = (A & 0x0F0F0F0Fu) | (((Bw >> sb0) << 4) & 0x30303030u) | (((C >> q0) << 6) & 0x40404040u) | e0;
  const uint32_t l1 = ((A >> 4) & 0x0F0F0F0Fu) | (((Bw >> (sb0 + 2)) << 4) & 0x30303030u) |
                      (((C >> (q0 + 1)) << 6) & 0x40404040u) | e1;
  w[0] = prmt(l0, h0, 0x5140);
  w[1] = prmt(l0, h0, 0x7362);
  w[2] = prmt(l1, h1, 0x5140);
  w[3] = prmt(l1, h1, 0x7362);
}

template <int SRC, int BT, int R, int MODE, bool FULL, int ADDR>
__device__ __forceinline__ void compute_chunk(const RegTable& t, const uint16_t* __restrict__ xc, int64_t K, int B,
                                              const ChunkBuf (&buf)[R], const bool (&live)[R], uint32_t vmask,
                                              int lane, float2 (&acc)[R][BT]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (!FULL && !((vmask >> i) & 1)) continue;
    uint32_t xw[BT][4];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      if (b < B) {
        const uint16_t* xb = xc + int64_t(b) * K + (ADDR == 2 ? 32 : 8) * lane;
        const uint4 v = ADDR == 2 ? (i == 0   ? ld_x_v4_at<0>(xb)
                                     : i == 1 ? ld_x_v4_at<16>(xb)
                                     : i == 2 ? ld_x_v4_at<32>(xb)
                                              : ld_x_v4_at<48>(xb))
                        : ADDR == 0 ? ld_x_v4(xb + kSlice * i)
                        : i == 0    ? ld_x_v4_at<0>(xb)
                        : i == 1    ? ld_x_v4_at<2 * kSlice>(xb)
                        : i == 2    ? ld_x_v4_at<4 * kSlice>(xb)
                                    : ld_x_v4_at<6 * kSlice>(xb);
        xw[b][0] = v.x; xw[b][1] = v.y; xw[b][2] = v.z; xw[b][3] = v.w;
      } else {
        xw[b][0] = xw[b][1] = xw[b][2] = xw[b][3] = 0u;
      }
    }
    float xf[MODE == 0 ? BT : 1][8];
    if (MODE == 0) {
#pragma unroll
      for (int b = 0; b < BT; ++b)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xf[MODE == 0 ? b : 0][2 * q] = bf16_lo(xw[b][q]);
          xf[MODE == 0 ? b : 0][2 * q + 1] = bf16_hi(xw[b][q]);
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (!live[j]) continue;
      uint32_t w[4];
      if (ADDR == 2 && SRC == kK15) {
        if (i == 0) group_slice_pairs_k15<0>(t, buf[j], w);
        else if (i == 1) group_slice_pairs_k15<1>(t, buf[j], w);
        else if (i == 2) group_slice_pairs_k15<2>(t, buf[j], w);
        else group_slice_pairs_k15<3>(t, buf[j], w);
      } else if (i == 0) slice_pairs<SRC, 0>(t, buf[j], lane, w);
      else if (i == 1) slice_pairs<SRC, 1>(t, buf[j], lane, w);
      else if (i == 2) slice_pairs<SRC, 2>(t, buf[j], lane, w);
      else slice_pairs<SRC, 3>(t, buf[j], lane, w);
#pragma unroll
      for (int b = 0; b < BT; ++b) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (MODE == 0)
            fma_wide(acc[j][b], w[q], xf[MODE == 0 ? b : 0][2 * q], xf[MODE == 0 ? b : 0][2 * q + 1]);
          else
            fma_mixed(acc[j][b], w[q], xw[b][q]);
        }
      }
    }
  }
}

template <int BT>
__device__ __forceinline__ void warp_reduce_store(float (&s)[BT], int B, float* __restrict__ y, int64_t N, int64_t r,
                                                  int lane) {
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    float v = s[b];
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && b < B) y[int64_t(b) * N + r] = v;
  }
}

// x * (w_true - w_placeholder) for one escape of the row starting at element rowbase.
template <int BT>
__device__ __forceinline__ void add_escape(const TensorDesc& d, const uint16_t* __restrict__ x, int B, uint64_t rowbase,
                                           uint32_t p, uint32_t val, float (&s)[BT]) {
  uint32_t wt, wph;
  if (d.scheme == WCOMP_BYTESPLIT) {
    wph = d.raw[p];
    wt = (val << 8) | wph;
  } else {
    wt = val;
    wph = val & 0x7Fu;
  }
  const float delta = __uint_as_float(wt << 16) - __uint_as_float(wph << 16);
  const int64_t k = int64_t(uint64_t(p) - rowbase);
#pragma unroll
  for (int b = 0; b < BT; ++b)
    if (b < B) s[b] = fmaf(__uint_as_float(uint32_t(x[int64_t(b) * d.K + k]) << 16), delta, s[b]);
}

__device__ __forceinline__ uint32_t load_esc_val(const TensorDesc& d, uint32_t e) {
  return d.scheme == WCOMP_BYTESPLIT ? uint32_t(d.esc_val[e]) : uint32_t(reinterpret_cast<const uint16_t*>(d.esc_val)[e]);
}

__device__ __forceinline__ uint32_t grab(uint32_t* slot, int lane) {
  uint32_t u = 0;
  if (lane == 0) u = atomicAdd(slot, 1u);
  return __shfl_sync(0xffffffffu, u, 0);
}

// ---------------------------------------------------------------------------
// The kernel (vector path: K % 32 == 0, aligned streams and x).
// ---------------------------------------------------------------------------
// One unit as the pipeline sees it.
template <int R>
struct UnitState {
  int ti;
  int64_t r0;
  uint32_t nchunks, vlast;
  uint32_t e_lo, e_hi;  // the unit's escapes: [e_lo, e_hi) of the tensor's escape list
  bool last_full;
  bool live[R];
};

template <int SRC, int R, bool AHEAD, int ADDR>
__device__ __forceinline__ void unit_state(const GemvBatch& p, uint32_t u, int lane, UnitState<R>& st, int start) {
  st.ti = owner(p.set_prefix, p.count, u, start);
  const TensorDesc& d = p.d[st.ti];
  st.r0 = int64_t(u - p.set_prefix[st.ti]) * R;
  st.nchunks = uint32_t(cdiv(uint64_t(d.K), kChunk));
  const uint32_t krem = uint32_t(d.K - int64_t(st.nchunks - 1) * kChunk);
  st.last_full = krem == kChunk;
  st.vlast = 0;
  if (ADDR == 2) {
    st.vlast = 32 * lane + 32 <= int(krem) ? 0xFu : 0u;  // the lane's group is whole or absent
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) st.vlast |= (kSlice * i + 8 * lane + 8 <= int(krem) ? 1u : 0u) << i;
  }
#pragma unroll
  for (int j = 0; j < R; ++j) st.live[j] = st.r0 + j < d.N;
  // requested one unit ahead, so the row index is at hand when the unit starts
  if (SRC != kPlain && AHEAD) {
    const int64_t r_end = st.r0 + R < d.N ? st.r0 + R : d.N;
    st.e_lo = d.row_index[st.r0];
    st.e_hi = d.row_index[r_end];
  } else {
    st.e_lo = st.e_hi = 0;
  }
}

// Row (j < R) of the unit and column of escape position `pos`; base is the
// unit's first element.  R is small, so this is R - 1 compares, no division.
template <int R>
__device__ __forceinline__ void esc_locate(uint32_t pos, uint64_t base, int64_t K, int& j, int64_t& k) {
  int64_t off = int64_t(uint64_t(pos) - base);
  j = 0;
#pragma unroll
  for (int jj = 1; jj < R; ++jj)
    if (off >= K) {
      off -= K;
      ++j;
    }
  k = off;
}

// x * (w_true - w_placeholder) for one escape: `lo` is the placeholder's low
// byte (byte-split; the escape value holds the high byte) and `val` the
// escape value (the whole word for K15).
template <int SCHEME>
__device__ __forceinline__ float esc_delta(uint32_t val, uint32_t lo) {
  uint32_t wt, wph;
  if (SCHEME == WCOMP_BYTESPLIT) {
    wph = lo;
    wt = (val << 8) | lo;
  } else {
    wt = val;
    wph = val & 0x7Fu;
  }
  return __uint_as_float(wt << 16) - __uint_as_float(wph << 16);
}

template <int SRC, int R, int ADDR>
__device__ __forceinline__ void load_unit_chunk(const GemvBatch& p, const UnitState<R>& st, uint32_t c, int lane,
                                                ChunkBuf (&bb)[R]) {
  const TensorDesc& d = p.d[st.ti];
  const Streams ss{d.codes, d.raw, d.pa, d.pb, d.pc};
  const bool full = c + 1 < st.nchunks || st.last_full;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (!st.live[j]) continue;
    const uint64_t eb = uint64_t(st.r0 + j) * uint64_t(d.K) + uint64_t(c) * kChunk;
    if (full) load_chunk<SRC, true, ADDR>(ss, eb, 0xF, lane, bb[j]);
    else load_chunk<SRC, false, ADDR>(ss, eb, st.vlast, lane, bb[j]);
  }
}

// How a unit finds its escapes' rows and the row index.  All three give the
// same sums; which one schedules best depends on the kernel's register
// budget, so each (scheme, batch) instantiation takes the one measured
// fastest.
enum EscMode {
  kEscDivide = 0,  // row index read when the unit starts; row of an escape by division
  kEscLocate = 1,  // row index read when the unit starts; row by R - 1 compares
  kEscAhead = 2,   // row index read one unit ahead; row by compares
};

#ifndef WCOMP_GEMV_ESC
#define WCOMP_GEMV_ESC -1  // -1: the table below; 0..2 forces one mode everywhere
#endif
// Address forms of the FMA kernel: 0 every slice address computed on its
// own, 1 per-chunk bases with immediate slice offsets, 2 one whole 32-element
// group per lane (one wide load per stream and compile-time K15 plane shifts,
// at the price of x loads strided by 64 bytes across lanes, which only pays
// at B = 1 and only for K15's heavier decode).
#ifndef WCOMP_GEMV_ADDR
#define WCOMP_GEMV_ADDR -1  // -1: the table below; 0..2 forces one form everywhere
#endif
constexpr int addr_mode(int src, int bt) {
  return WCOMP_GEMV_ADDR >= 0 ? WCOMP_GEMV_ADDR : src == kPlain ? 0 : src == kK15 && bt == 1 ? 2 : 1;
}

constexpr int esc_mode(int src, int bt) {
  return WCOMP_GEMV_ESC >= 0 ? WCOMP_GEMV_ESC
         : src == kBytesplit ? (bt == 1 ? kEscDivide : bt == 2 ? kEscLocate : bt <= 8 ? kEscAhead : kEscLocate)
         : src == kK15       ? (bt == 1 ? kEscLocate : bt == 2 ? kEscAhead : bt == 4 ? kEscDivide
                                : bt == 8 ? kEscAhead : kEscLocate)
                             : kEscLocate;
}

// The kernel (vector path: K % 32 == 0, aligned streams and x).  The warp
// runs one continuous pipeline over (unit, chunk) items: while it computes an
// item, the next item's loads are in flight, including across the boundary
// between units, so no unit starts with an exposed load latency.
template <int SRC, int BT, int R, int MINB, int MODE, int ESC>
__global__ void __launch_bounds__(kThreads, MINB)
    gemv_kernel(const __grid_constant__ GemvBatch p, uint32_t total_units, int B, uint32_t* __restrict__ slot) {
  const int lane = threadIdx.x & 31;
  constexpr bool kAhead = ESC == kEscAhead;
  constexpr int kAddr = addr_mode(SRC, BT);
  uint32_t u = grab(slot, lane);
  if (u < total_units) {
    uint32_t u_next = grab(slot, lane);
    UnitState<R> cur, nxt;
    unit_state<SRC, R, kAhead, kAddr>(p, u, lane, cur, 0);
    // load cursor: the item after the one being computed
    ChunkBuf b0[R], b1[R];
    load_unit_chunk<SRC, R, kAddr>(p, cur, 0, lane, b0);
    float2 acc[R][BT];
    uint32_t p0 = 0, v0 = 0;
    auto begin_unit = [&]() {
#pragma unroll
      for (int j = 0; j < R; ++j)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[j][b] = make_float2(0.f, 0.f);
      if (SRC != kPlain) {
        const TensorDesc& d = p.d[cur.ti];
        if (!kAhead) {
          const int64_t r_end = cur.r0 + R < d.N ? cur.r0 + R : d.N;
          cur.e_lo = d.row_index[cur.r0];
          cur.e_hi = d.row_index[r_end];
        }
        if (cur.e_lo + lane < cur.e_hi) {
          p0 = d.esc_pos[cur.e_lo + lane];
          v0 = load_esc_val(d, cur.e_lo + lane);
        }
      }
    };
    auto end_unit = [&]() {
      const TensorDesc& d = p.d[cur.ti];
      const int64_t K = d.K;
      float s[R][BT];
#pragma unroll
      for (int j = 0; j < R; ++j)
#pragma unroll
        for (int b = 0; b < BT; ++b) s[j][b] = acc[j][b].x + acc[j][b].y;
      if (SRC != kPlain) {
        const uint16_t* __restrict__ x = p.x[cur.ti];
        const uint64_t base = uint64_t(cur.r0) * uint64_t(K);
        for (uint32_t e = cur.e_lo + lane; e < cur.e_hi; e += 32) {
          uint32_t pos = p0, val = v0;
          if (e != cur.e_lo + lane) {
            pos = d.esc_pos[e];
            val = load_esc_val(d, e);
          }
          int j;
          int64_t k;
          if (ESC == kEscDivide) {
            j = int(int64_t(pos / uint64_t(K)) - cur.r0);
            k = int64_t(uint64_t(pos) - base) - int64_t(j) * K;
          } else {
            esc_locate<R>(pos, base, K, j, k);
          }
          const uint32_t lo = SRC == kBytesplit ? uint32_t(d.raw[pos]) : 0u;
          const float delta = esc_delta<SRC == kBytesplit ? WCOMP_BYTESPLIT : WCOMP_K15>(val, lo);
#pragma unroll
          for (int jj = 0; jj < R; ++jj) {
            if (jj != j) continue;
#pragma unroll
            for (int b = 0; b < BT; ++b)
              if (b < B) s[jj][b] = fmaf(__uint_as_float(uint32_t(x[int64_t(b) * K + k]) << 16), delta, s[jj][b]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (cur.live[j]) warp_reduce_store<BT>(s[j], B, p.y[cur.ti], d.N, cur.r0 + j, lane);
    };
    auto compute = [&](uint32_t c, const ChunkBuf (&bb)[R]) {
      const TensorDesc& d = p.d[cur.ti];
      const uint16_t* xc = p.x[cur.ti] + uint64_t(c) * kChunk;
      if (c + 1 < cur.nchunks || cur.last_full)
        compute_chunk<SRC, BT, R, MODE, true, kAddr>(d.t, xc, d.K, B, bb, cur.live, 0xF, lane, acc);
      else
        compute_chunk<SRC, BT, R, MODE, false, kAddr>(d.t, xc, d.K, B, bb, cur.live, cur.vlast, lane, acc);
    };
    begin_unit();
    // position of the item held in the "current" buffer
    uint32_t c = 0;
    bool have_next_unit = u_next < total_units;
    if (have_next_unit) unit_state<SRC, R, kAhead, kAddr>(p, u_next, lane, nxt, cur.ti);
    // One step: request the item after (cur, c) into `ld`, compute (cur, c)
    // from `cb`, then advance.  Returns false when nothing is left.
    auto step = [&](ChunkBuf (&cb)[R], ChunkBuf (&ld)[R]) -> bool {
      const bool last_of_unit = c + 1 == cur.nchunks;
      if (!last_of_unit) load_unit_chunk<SRC, R, kAddr>(p, cur, c + 1, lane, ld);
      else if (have_next_unit) load_unit_chunk<SRC, R, kAddr>(p, nxt, 0, lane, ld);
      compute(c, cb);
      if (!last_of_unit) {
        ++c;
        return true;
      }
      end_unit();
      if (!have_next_unit) return false;
      cur = nxt;
      c = 0;
      begin_unit();
      u_next = grab(slot, lane);
      have_next_unit = u_next < total_units;
      if (have_next_unit) unit_state<SRC, R, kAhead, kAddr>(p, u_next, lane, nxt, cur.ti);
      return true;
    };
    while (step(b0, b1) && step(b1, b0)) {
    }
  }
  // The last warp to finish returns the counter slot to zero for the next launch.
  if (lane == 0) {
    __threadfence();
    const uint32_t total_warps = gridDim.x * kWarps;
    if (atomicAdd(slot + 1, 1u) == total_warps - 1) {
      atomicExch(slot, 0u);
      atomicExch(slot + 1, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// The staged kernel: the same work decomposition, with the weight streams
// brought into shared memory by bulk asynchronous copies (TMA, 1-D form).
//
// Every warp owns a ring of S stages.  One stage holds one 1024-element chunk
// of each of the unit's R rows; lane 0 keeps S chunks in flight (it grabs the
// next unit as soon as the current one is fully requested, so the ring runs
// across unit boundaries) and every lane waits on the stage's mbarrier before
// reading its slices out of shared memory.  Bytes in flight per SM no longer
// cost registers, so far more of them are outstanding than with register
// double buffering.  Waits are bounded: a stage that never completes sets the
// device error word and the warp stops after draining its own copies.
// ---------------------------------------------------------------------------
constexpr uint32_t kWaitLimit = 1u << 27;  // polls before giving up (well over a second)

template <int SRC>
struct Geom {
  // shared-memory bytes for one row's chunk: codes | raw   (byte-split)
  //                                          codes | A | B window | C window   (K15)
  //                                          BF16 values   (plain)
  static constexpr uint32_t kB = 1024;                     // K15 plane B window offset
  static constexpr uint32_t kC = 1024 + 256 + 16;          // K15 plane C window offset
  static constexpr uint32_t row_bytes = SRC == kBytesplit ? 1536 : SRC == kK15 ? (kC + 128 + 16) : 2048;
};

// Words of slice i of one row, read from a stage.
struct SliceWords {
  uint32_t cw, r0, r1, A, Bw, C;
  uint4 pw;
};

template <int SRC>
__device__ __forceinline__ SliceWords read_slice(const uint8_t* rowbuf, int i, int lane, uint32_t dB, uint32_t dC) {
  SliceWords w;
  if (SRC == kPlain) {
    w.pw = *reinterpret_cast<const uint4*>(rowbuf + 512 * i + 16 * lane);
    return w;
  }
  w.cw = *reinterpret_cast<const uint32_t*>(rowbuf + 128 * i + 4 * lane);
  if (SRC == kBytesplit) {
    const uint2 r = *reinterpret_cast<const uint2*>(rowbuf + 512 + 256 * i + 8 * lane);
    w.r0 = r.x;
    w.r1 = r.y;
  } else {
    w.A = *reinterpret_cast<const uint32_t*>(rowbuf + 512 + 128 * i + 4 * lane);
    w.Bw = *reinterpret_cast<const uint32_t*>(rowbuf + Geom<kK15>::kB + dB + 64 * i + 8 * (lane >> 2) +
                                              4 * ((lane >> 1) & 1));
    w.C = *reinterpret_cast<const uint32_t*>(rowbuf + Geom<kK15>::kC + dC + 32 * i + 4 * (lane >> 2));
  }
  return w;
}

template <int SRC>
__device__ __forceinline__ void words_to_pairs(const RegTable& t, const SliceWords& sw, int lane, uint32_t (&w)[4]) {
  if (SRC == kPlain) {
    w[0] = sw.pw.x; w[1] = sw.pw.y; w[2] = sw.pw.z; w[3] = sw.pw.w;
    return;
  }
  const QuadMasks m = code_masks(sw.cw);
  const uint32_t m7 = sw.cw & 0x77777777u;
  uint32_t h0, h1, l0, l1;
  lookup8(t.hi, m7, m, h0, h1);
  if (SRC == kBytesplit) {
    l0 = sw.r0;
    l1 = sw.r1;
  } else {
    const uint32_t q0 = 2 * (lane & 3), sb0 = 4 * (lane & 1);
    uint32_t e0, e1;
    lookup8(t.e0, m7, m, e0, e1);
    l0 = (sw.A & 0x0F0F0F0Fu) | (((sw.Bw >> sb0) << 4) & 0x30303030u) | (((sw.C >> q0) << 6) & 0x40404040u) | e0;
    l1 = ((sw.A >> 4) & 0x0F0F0F0Fu) | (((sw.Bw >> (sb0 + 2)) << 4) & 0x30303030u) |
         (((sw.C >> (q0 + 1)) << 6) & 0x40404040u) | e1;
  }
  w[0] = prmt(l0, h0, 0x5140);
  w[1] = prmt(l0, h0, 0x7362);
  w[2] = prmt(l1, h1, 0x5140);
  w[3] = prmt(l1, h1, 0x7362);
}

// Issue the bulk copies of chunk c of unit u's rows into one stage.
template <int SRC, int R>
__device__ __forceinline__ void issue_chunk(const GemvBatch& p, uint32_t u, uint32_t c, uint8_t* stage,
                                            uint64_t* bar) {
  const int ti = owner(p.set_prefix, p.count, u);
  const TensorDesc& d = p.d[ti];
  const int64_t r0 = int64_t(u - p.set_prefix[ti]) * R;
  const uint64_t K = uint64_t(d.K);
  const uint64_t k0 = uint64_t(c) * kChunk;
  const uint32_t len = uint32_t(K - k0 < uint64_t(kChunk) ? K - k0 : uint64_t(kChunk));
  uint32_t bytes = 0;
  uint32_t sz[R][4];
  const uint8_t* src[R][4];
#pragma unroll
  for (int j = 0; j < R; ++j) {
#pragma unroll
    for (int q = 0; q < 4; ++q) sz[j][q] = 0;
    if (r0 + j >= d.N) continue;
    const uint64_t e0 = uint64_t(r0 + j) * K + k0;
    if (SRC == kBytesplit) {
      src[j][0] = d.codes + e0 / 2; sz[j][0] = len / 2;
      src[j][1] = d.raw + e0; sz[j][1] = len;
    } else if (SRC == kK15) {
      src[j][0] = d.codes + e0 / 2; sz[j][0] = len / 2;
      src[j][1] = d.pa + e0 / 2; sz[j][1] = len / 2;
      const uint64_t bs = (e0 / 4) & ~uint64_t(15), be = ((e0 + len) / 4 + 15) & ~uint64_t(15);
      src[j][2] = d.pb + bs; sz[j][2] = uint32_t(be - bs);
      const uint64_t cs = (e0 / 8) & ~uint64_t(15), ce = ((e0 + len) / 8 + 15) & ~uint64_t(15);
      src[j][3] = d.pc + cs; sz[j][3] = uint32_t(ce - cs);
    } else {
      src[j][0] = d.raw + 2 * e0; sz[j][0] = 2 * len;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) bytes += sz[j][q];
  }
#if WCOMP_GEMV_PROXY_FENCE
  fence_proxy_async();  // earlier generic reads of this stage come before the new async writes
#endif
  mbar_expect_tx(bar, bytes);
#pragma unroll
  for (int j = 0; j < R; ++j) {
    uint8_t* rb = stage + j * Geom<SRC>::row_bytes;
    const uint32_t dst_off[4] = {0u, SRC == kBytesplit || SRC == kK15 ? 512u : 0u, Geom<kK15>::kB, Geom<kK15>::kC};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (sz[j][q]) bulk_load(rb + dst_off[q], src[j][q], sz[j][q], bar);
  }
}

template <int SRC, int BT, int R, int MODE, int S, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    gemv_tma_kernel(const __grid_constant__ GemvBatch p, uint32_t total_units, int B, uint32_t* __restrict__ slot,
                    uint32_t* __restrict__ err) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr uint32_t kStage = (R * Geom<SRC>::row_bytes + 127) & ~127u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* ring = smem + uint32_t(warp) * (S * kStage + S * 8 + 2 * S * 4);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + S * kStage);
  uint32_t* uq = reinterpret_cast<uint32_t*>(ring + S * kStage + S * 8);
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // producer state (warp-uniform): next unit / chunk to request; the unit
  // after it is grabbed one unit ahead so the atomic's latency stays hidden
  uint32_t pu = grab(slot, lane), pc = 0, pseq = 0;
  uint32_t pu_next = grab(slot, lane);
  uint32_t issued = 0, consumed = 0;
  auto chunks_of = [&](uint32_t u) -> uint32_t {
    const int ti = owner(p.set_prefix, p.count, u);
    return uint32_t(cdiv(uint64_t(p.d[ti].K), kChunk));
  };
  uint32_t pn = pu < total_units ? chunks_of(pu) : 0;
  // consumer state
  uint32_t cseq = 0, cu = 0, cc = 0, cn = 0;
  int ti = 0;
  int64_t r0 = 0;
  bool live[R];
  float2 acc[R][BT];
  uint32_t e_lo = 0, e_hi = 0, p0 = 0, v0 = 0;
  bool failed = false;

  while (true) {
    // keep S chunks requested
    while (pu < total_units && issued - consumed < uint32_t(S)) {
      if (pc == 0) {
        if (lane == 0) uq[pseq % (2 * S)] = pu;
        ++pseq;
      }
      if (lane == 0) issue_chunk<SRC, R>(p, pu, pc, ring + (issued % S) * kStage, &bars[issued % S]);
      ++issued;
      if (++pc == pn) {
        pu = pu_next;
        pc = 0;
        pn = pu < total_units ? chunks_of(pu) : 0;
        if (pu < total_units) pu_next = grab(slot, lane);
      }
    }
    __syncwarp();
    if (consumed == issued) break;
    if (cc == 0) {  // start a unit
      cu = uq[cseq % (2 * S)];
      ++cseq;
      ti = owner(p.set_prefix, p.count, cu);
      const TensorDesc& d = p.d[ti];
      r0 = int64_t(cu - p.set_prefix[ti]) * R;
      cn = uint32_t(cdiv(uint64_t(d.K), kChunk));
#pragma unroll
      for (int j = 0; j < R; ++j) live[j] = r0 + j < d.N;
#pragma unroll
      for (int j = 0; j < R; ++j)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[j][b] = make_float2(0.f, 0.f);
      if (SRC != kPlain) {
        const int64_t r_end = r0 + R < d.N ? r0 + R : d.N;
        e_lo = d.row_index[r0];
        e_hi = d.row_index[r_end];
        if (e_lo + lane < e_hi) {
          p0 = d.esc_pos[e_lo + lane];
          v0 = load_esc_val(d, e_lo + lane);
        }
      }
    }
    const TensorDesc& d = p.d[ti];
    const int64_t K = d.K;
    const uint32_t st = consumed % S;
    if (!mbar_wait(&bars[st], (consumed / S) & 1, kWaitLimit)) {
      failed = true;
      break;
    }
    // compute chunk cc of the current unit
    {
      const uint64_t k0 = uint64_t(cc) * kChunk;
      const uint32_t len = uint32_t(uint64_t(K) - k0 < uint64_t(kChunk) ? uint64_t(K) - k0 : uint64_t(kChunk));
      const uint16_t* xc = p.x[ti] + k0;
      const uint8_t* sbuf = ring + st * kStage;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool valid = kSlice * i + 8 * lane + 8 <= int(len);
        if (len == kChunk || valid) {
          uint32_t xw[BT][4];
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            if (b < B) {
              const uint4 v = ld_x_v4(xc + int64_t(b) * K + kSlice * i + 8 * lane);
              xw[b][0] = v.x; xw[b][1] = v.y; xw[b][2] = v.z; xw[b][3] = v.w;
            } else {
              xw[b][0] = xw[b][1] = xw[b][2] = xw[b][3] = 0u;
            }
          }
          float xf[MODE == 0 ? BT : 1][8];
          if (MODE == 0) {
#pragma unroll
            for (int b = 0; b < BT; ++b)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                xf[MODE == 0 ? b : 0][2 * q] = bf16_lo(xw[b][q]);
                xf[MODE == 0 ? b : 0][2 * q + 1] = bf16_hi(xw[b][q]);
              }
          }
#pragma unroll
          for (int j = 0; j < R; ++j) {
            if (!live[j]) continue;
            uint32_t dB = 0, dC = 0;
            if (SRC == kK15) {
              const uint64_t e0 = uint64_t(r0 + j) * uint64_t(K) + k0;
              dB = uint32_t((e0 / 4) & 15);
              dC = uint32_t((e0 / 8) & 15);
            }
            const SliceWords sw = read_slice<SRC>(sbuf + j * Geom<SRC>::row_bytes, i, lane, dB, dC);
            uint32_t w[4];
            words_to_pairs<SRC>(d.t, sw, lane, w);
#pragma unroll
            for (int b = 0; b < BT; ++b)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (MODE == 0)
                  fma_wide(acc[j][b], w[q], xf[MODE == 0 ? b : 0][2 * q], xf[MODE == 0 ? b : 0][2 * q + 1]);
                else
                  fma_mixed(acc[j][b], w[q], xw[b][q]);
              }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with the stage before lane 0 refills it
    ++consumed;
    if (++cc == cn) {  // unit complete: escapes, reduction, store
      cc = 0;
      float s[R][BT];
#pragma unroll
      for (int j = 0; j < R; ++j)
#pragma unroll
        for (int b = 0; b < BT; ++b) s[j][b] = acc[j][b].x + acc[j][b].y;
      if (SRC != kPlain) {
        const uint16_t* __restrict__ x = p.x[ti];
        for (uint32_t e = e_lo + lane; e < e_hi; e += 32) {
          uint32_t pos = p0, val = v0;
          if (e != e_lo + lane) {
            pos = d.esc_pos[e];
            val = load_esc_val(d, e);
          }
          const int64_t j = int64_t(pos / uint64_t(K)) - r0;
#pragma unroll
          for (int jj = 0; jj < R; ++jj)
            if (jj == j) add_escape<BT>(d, x, B, uint64_t(r0 + jj) * uint64_t(K), pos, val, s[jj]);
        }
      }
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (live[j]) warp_reduce_store<BT>(s[j], B, p.y[ti], d.N, r0 + j, lane);
    }
  }
  if (failed) {
    // record the failure and let this warp's own copies land before exiting
    if (lane == 0) atomicOr(err, 1u);
    for (uint32_t k = consumed + 1; k < issued; ++k) mbar_wait(&bars[k % S], (k / S) & 1, kWaitLimit);
    __syncwarp();
  }
  // The last warp to finish returns the counter slot to zero for the next launch.
  if (lane == 0) {
    __threadfence();
    const uint32_t total_warps = gridDim.x * kWarps;
    if (atomicAdd(slot + 1, 1u) == total_warps - 1) {
      atomicExch(slot, 0u);
      atomicExch(slot + 1, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core path (mma.sync m16n8k16, BF16 in, fp32 accumulate).
//
// For larger batches the per-element fp32 FMAs and the x reads through L1
// bound the kernel above, not HBM.  Here one warp-level MMA takes 16 batch
// rows (M; the batch padded to 8 or 16) against 8 weight rows (N) over 16
// elements of K, so the multiply costs one instruction per 128 weights of a
// warp and x is read once per 8 weight rows.
//
// Work unit: 8 consecutive rows of one tensor.  A CTA of 4 warps takes a unit
// and splits its K range into 4 contiguous runs of 128-element k-blocks; the
// warps' partial 16x8 tiles are summed in shared memory in a fixed order.
//
// Lane (g = lane >> 2, t = lane & 3) holds weight row g of the unit and, in
// k-block kb, its elements 128 kb + 32 t .. +31: one whole 32-element group,
// fetched with one wide load per stream (16 bytes of codes, 32 of raw bytes),
// so a warp's request for a stream is 8 row segments of 64 or 128 bytes.  The
// lane decodes its group as four slices of 8 (slice i = elements 8i .. 8i+7).
// The MMA's k order inside a step is a relabelling: step s = 2 i + h pairs
// the lane's elements 8i + 4h .. +3 with the B-fragment rows 2t, 2t+1, 2t+8,
// 2t+9 and the same x elements with the A-fragment columns, which leaves the
// sum unchanged.
//
// Escapes: the tile sums the placeholders; after the k-blocks, thread
// (row j, batch b, part q) adds x[b, k] * (w_true - w_placeholder) over the
// q-th share of row j's escapes, and the parts are summed in a fixed order.
// ---------------------------------------------------------------------------
#ifndef WCOMP_GEMV_MMA_WARPS
#define WCOMP_GEMV_MMA_WARPS 8
#endif
constexpr int kMmaWarps = WCOMP_GEMV_MMA_WARPS;  // warps splitting one unit's K range
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kKBlock = 128;
// The escape corrections give every (row, batch) pair of a unit at least one
// thread (8 rows x 16 batches) and the final sums one thread per output.
static_assert(kMmaThreads >= 8 * 16 && kMmaThreads % (8 * 16) == 0, "MMA CTA too small for 8 rows x 16 batches");

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A unit as the tensor-core kernel sees it.
struct MmaUnit {
  int ti;
  int64_t r0;
  int rows;          // valid rows (1..8)
  uint32_t kb0, kb1;  // this warp's k-blocks [kb0, kb1)
  uint32_t kvalid;   // valid elements of the tensor's last k-block (32..128)
  uint32_t nkb;      // k-blocks per row
};

// The k-block range of this warp, derived from the tensor's K.
__device__ __forceinline__ void mma_unit_range(const GemvBatch& p, int warp, MmaUnit& m) {
  const TensorDesc& d = p.d[m.ti];
  m.nkb = uint32_t(cdiv(uint64_t(d.K), kKBlock));
  m.kvalid = uint32_t(d.K - int64_t(m.nkb - 1) * kKBlock);
  m.kb0 = uint32_t(uint64_t(m.nkb) * warp / kMmaWarps);
  m.kb1 = uint32_t(uint64_t(m.nkb) * (warp + 1) / kMmaWarps);
}

// Tensor, first row and rows of unit u (the range is filled in separately,
// so a unit held for later costs three values, not seven).
__device__ __forceinline__ void mma_unit(const GemvBatch& p, uint32_t u, int start, MmaUnit& m) {
  m.ti = owner(p.set_prefix, p.count, u, start);
  const TensorDesc& d = p.d[m.ti];
  m.r0 = int64_t(u - p.set_prefix[m.ti]) * 8;
  m.rows = int(d.N - m.r0 < 8 ? d.N - m.r0 : 8);
}

// Loads of k-block kb of unit m for this lane: row g, elements 32 t .. +31 of
// the k-block, one wide load per stream.  Lanes whose row is past N or whose
// quarter is past K load nothing.  The lane's first element is a multiple of
// 32 (K % 32 == 0), so every load is aligned to its width.
//   byte-split: v[0..3] codes, v[4..11] raw bytes
//   K15:        v[0..3] codes, v[4..7] plane A, v[8..9] plane B, v[12] plane C
//   plain:      v[0..15] the 32 BF16 values
template <int SRC>
__device__ __forceinline__ void load_kblock(const GemvBatch& p, const MmaUnit& m, uint32_t kb, int g, int t,
                                            ChunkBuf& b) {
  if (g >= m.rows) return;
  const uint32_t valid = kb + 1 == m.nkb ? m.kvalid : uint32_t(kKBlock);
  if (uint32_t(32 * t) >= valid) return;
  const TensorDesc& d = p.d[m.ti];
  const uint64_t e = uint64_t(m.r0 + g) * uint64_t(d.K) + uint64_t(kb) * kKBlock + 32 * t;
  if (SRC == kPlain) {
    uint32_t r[8];
    ld_stream_v8(d.raw + 2 * e, r);
#pragma unroll
    for (int k = 0; k < 8; ++k) b.v[k] = r[k];
    ld_stream_v8(d.raw + 2 * e + 32, r);
#pragma unroll
    for (int k = 0; k < 8; ++k) b.v[8 + k] = r[k];
    return;
  }
  const uint4 c = ld_stream_v4(d.codes + (e >> 1));
  b.v[0] = c.x; b.v[1] = c.y; b.v[2] = c.z; b.v[3] = c.w;
  if (SRC == kBytesplit) {
    uint32_t r[8];
    ld_stream_v8(d.raw + e, r);
#pragma unroll
    for (int k = 0; k < 8; ++k) b.v[4 + k] = r[k];
  } else {
    const uint4 a = ld_stream_v4(d.pa + (e >> 1));
    b.v[4] = a.x; b.v[5] = a.y; b.v[6] = a.z; b.v[7] = a.w;
    const uint2 bb = ld_stream_v2(d.pb + (e >> 2));
    b.v[8] = bb.x; b.v[9] = bb.y;
    b.v[12] = ld_stream_u32(d.pc + (e >> 3));
  }
}

// One k-block: decode each slice into B fragments and issue its two MMAs.
template <int SRC, int XB>
__device__ __forceinline__ void mma_kblock(const RegTable& tab, const uint16_t* __restrict__ x, int64_t K, int B,
                                           const MmaUnit& m, uint32_t kb, int lane, const ChunkBuf& b,
                                           float (&acc)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t valid = kb + 1 == m.nkb ? m.kvalid : uint32_t(kKBlock);
  const bool live = uint32_t(32 * t) < valid;
  const bool wlive = live && g < m.rows;
  const uint16_t* xg = x + int64_t(g) * K + int64_t(kb) * kKBlock + 32 * t;
  const uint16_t* xg8 = xg + 8 * K;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (wlive) {
      if (SRC == kK15) {
        if (i == 0) group_slice_pairs_k15<0>(tab, b, w);
        else if (i == 1) group_slice_pairs_k15<1>(tab, b, w);
        else if (i == 2) group_slice_pairs_k15<2>(tab, b, w);
        else group_slice_pairs_k15<3>(tab, b, w);
      } else {
        if (i == 0) slice_pairs<SRC, 0>(tab, b, lane, w);
        else if (i == 1) slice_pairs<SRC, 1>(tab, b, lane, w);
        else if (i == 2) slice_pairs<SRC, 2>(tab, b, lane, w);
        else slice_pairs<SRC, 3>(tab, b, lane, w);
      }
    }
    uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = make_uint4(0u, 0u, 0u, 0u);
    if (live && g < B) xa = ld_x_v4(xg + 8 * i);
    if (XB == 16 && live && g + 8 < B) xb = ld_x_v4(xg8 + 8 * i);
    mma_bf16(acc, xa.x, xb.x, xa.y, xb.y, w[0], w[1]);
    mma_bf16(acc, xa.z, xb.z, xa.w, xb.w, w[2], w[3]);
  }
}

// x transposed for the escape corrections: xt[i][k * XB + b] = x_i[b, k]
// (zero for b >= B), so one thread reads every batch value of column k of
// tensor i with one or two 16-byte loads.
struct XtBatch {
  uint16_t* p[kMaxBatch];
  uint32_t kprefix[kMaxBatch + 1];  // first column of each tensor in the grid
  int count;
};

template <int XW>
__global__ void __launch_bounds__(256) transpose_x_kernel(const __grid_constant__ GemvBatch b,
                                                          const __grid_constant__ XtBatch xt, int B) {
  static_assert(XW == 2 || XW == 4 || XW == 8 || XW == 16, "transposed width");
  const uint32_t total = xt.kprefix[xt.count];
  for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < total; c += gridDim.x * blockDim.x) {
    int i = 0;
    while (i + 1 < xt.count && xt.kprefix[i + 1] <= c) ++i;
    const int64_t K = b.d[i].K;
    const uint32_t k = c - xt.kprefix[i];
    const uint16_t* x = b.x[i];
    uint32_t v[XW / 2];
#pragma unroll
    for (int q = 0; q < XW / 2; ++q) {
      const uint32_t lo = 2 * q < B ? uint32_t(x[int64_t(2 * q) * K + k]) : 0u;
      const uint32_t hi = 2 * q + 1 < B ? uint32_t(x[int64_t(2 * q + 1) * K + k]) : 0u;
      v[q] = lo | (hi << 16);
    }
    uint16_t* out = xt.p[i] + uint64_t(k) * XW;
    if (XW == 2) {
      *reinterpret_cast<uint32_t*>(out) = v[0];
    } else if (XW == 4) {
      *reinterpret_cast<uint2*>(out) = make_uint2(v[0], v[1 % (XW / 2)]);
    } else {
#pragma unroll
      for (int q = 0; q < XW / 8; ++q)
        reinterpret_cast<uint4*>(out)[q] = make_uint4(v[(4 * q) % (XW / 2)], v[(4 * q + 1) % (XW / 2)],
                                                      v[(4 * q + 2) % (XW / 2)], v[(4 * q + 3) % (XW / 2)]);
    }
  }
}

template <int SRC, int XB, int MINB, int XW = 0>
__global__ void __launch_bounds__(kMmaThreads, MINB)
    gemv_mma_kernel(const __grid_constant__ GemvBatch p, uint32_t total_units, int B, uint32_t* __restrict__ slot,
                    const __grid_constant__ XtBatch xt) {
  // Two sets, alternating by unit parity, so one barrier per unit suffices:
  // a set is rewritten two units later, after every thread has passed the
  // next unit's barrier and so finished reading it.
  __shared__ float part[2][kMmaWarps][32][4];
  // per-thread corrections (x gathered per batch row), or with XT per-warp
  // sums for every (batch, row) of the unit
  constexpr bool XT = XW > 0;  // corrections from x transposed to [K][XW]
  __shared__ float corr[2][XT ? kMmaWarps * 16 * 8 : kMmaThreads];
  __shared__ uint32_t first_unit, next_unit[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  if (threadIdx.x == 0) {
    first_unit = atomicAdd(slot, 1u);
    next_unit[1] = atomicAdd(slot, 1u);
  }
  __syncthreads();
  // This thread's share of the escape corrections: row cj, batch cb, part cq
  // of cP (cbp batch slots, cP = threads / (8 cbp) parts per (row, batch)).
  const int cbp = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
  const int cP = kMmaThreads / (8 * cbp);
  const int cj = threadIdx.x & 7, cb = (threadIdx.x >> 3) % cbp, cq = (threadIdx.x >> 3) / cbp;
  uint32_t u = first_unit, u_next = next_unit[1];
  if (u < total_units) {
    MmaUnit cur, nxt;
    uint32_t ce0 = 0, ce1 = 0, ne0 = 0, ne1 = 0;  // row cj's escapes in the current / next unit
    auto row_escapes = [&](const MmaUnit& m, uint32_t& e0, uint32_t& e1) {
      if (SRC == kPlain || cj >= m.rows) return;
      const TensorDesc& d = p.d[m.ti];
      e0 = d.row_index[m.r0 + cj];
      e1 = d.row_index[m.r0 + cj + 1];
    };
    mma_unit(p, u, 0, cur);
    mma_unit_range(p, warp, cur);
    row_escapes(cur, ce0, ce1);
    bool have_next = u_next < total_units;
    if (have_next) {
      mma_unit(p, u_next, cur.ti, nxt);
      row_escapes(nxt, ne0, ne1);
    }
    ChunkBuf b0, b1;
    uint32_t kb = cur.kb0;
    if (kb < cur.kb1) load_kblock<SRC>(p, cur, kb, g, t, b0);
    float acc[4];
    int par = 0;
    uint32_t grabbed = 0;
    // This thread's first escape of the unit: position and value requested
    // when the unit starts, its low byte and x value one k-block later, so the
    // correction after the unit's barrier does not wait on a dependent load.
    // Byte-split with 8 batch rows only: with 16 batch rows the extra live
    // registers spill, and K15's many escapes per thread gain nothing from
    // prefetching one (both measured slower).
    constexpr bool kFirst = SRC == kBytesplit && XB == 8;
    uint32_t f_pos = 0, f_val = 0, f_lo = 0, f_x = 0, steps_in_unit = 0;
    bool f_ready = false;
    auto request_first = [&]() {
      f_ready = false;
      steps_in_unit = 0;
      if (!kFirst || cj >= cur.rows || cb >= B || ce0 + cq >= ce1) return;
      const TensorDesc& d = p.d[cur.ti];
      f_pos = d.esc_pos[ce0 + cq];
      f_val = load_esc_val(d, ce0 + cq);
    };
    auto fetch_first = [&]() {
      f_ready = true;
      if (!kFirst || cj >= cur.rows || cb >= B || ce0 + cq >= ce1) return;
      const TensorDesc& d = p.d[cur.ti];
      const uint64_t rowbase = uint64_t(cur.r0 + cj) * uint64_t(d.K);
      f_lo = SRC == kBytesplit ? uint32_t(d.raw[f_pos]) : 0u;
      f_x = uint32_t(p.x[cur.ti][int64_t(cb) * d.K + int64_t(uint64_t(f_pos) - rowbase)]);
    };
    request_first();
    if (threadIdx.x == 0) grabbed = atomicAdd(slot, 1u);
    auto unit_end = [&]() {
      // partial tiles, escape corrections, fixed-order sums
      const TensorDesc& d = p.d[cur.ti];
      part[par][warp][lane][0] = acc[0];
      part[par][warp][lane][1] = acc[1];
      part[par][warp][lane][2] = acc[2];
      part[par][warp][lane][3] = acc[3];
      if constexpr (XT) {
        // thread (row j = cj, part q = tid / 8 of 32): every batch row at once
        // from the transposed x; the four parts of a warp are summed by a
        // fixed shuffle tree, the warps in order in the final sum
        constexpr int W = XT ? XW : 1;
        float cs[W];
#pragma unroll
        for (int b = 0; b < W; ++b) cs[b] = 0.f;
        if (cj < cur.rows) {
          const uint64_t rowbase = uint64_t(cur.r0 + cj) * uint64_t(d.K);
          const uint16_t* xtb = xt.p[cur.ti];
          for (uint32_t e = ce0 + (threadIdx.x >> 3); e < ce1; e += kMmaThreads / 8) {
            const uint32_t pos = d.esc_pos[e];
            const float delta = esc_delta<SRC == kBytesplit ? WCOMP_BYTESPLIT : WCOMP_K15>(
                load_esc_val(d, e), SRC == kBytesplit ? uint32_t(d.raw[pos]) : 0u);
            const uint16_t* xr = xtb + uint64_t(uint64_t(pos) - rowbase) * W;
            uint32_t wv[W / 2 > 0 ? W / 2 : 1];
            if (W == 2) {
              wv[0] = *reinterpret_cast<const uint32_t*>(xr);
            } else if (W == 4) {
              const uint2 v = *reinterpret_cast<const uint2*>(xr);
              wv[0] = v.x;
              wv[1 % (W / 2 > 0 ? W / 2 : 1)] = v.y;
            } else {
#pragma unroll
              for (int q = 0; q < W / 8; ++q) {
                const uint4 v = reinterpret_cast<const uint4*>(xr)[q];
                wv[4 * q] = v.x; wv[4 * q + 1] = v.y; wv[4 * q + 2] = v.z; wv[4 * q + 3] = v.w;
              }
            }
#pragma unroll
            for (int h = 0; h < W / 2; ++h) {
              cs[2 * h] = fmaf(bf16_lo(wv[h]), delta, cs[2 * h]);
              cs[2 * h + 1] = fmaf(bf16_hi(wv[h]), delta, cs[2 * h + 1]);
            }
          }
        }
#pragma unroll
        for (int b = 0; b < W; ++b) {
          cs[b] += __shfl_xor_sync(0xffffffffu, cs[b], 8);
          cs[b] += __shfl_xor_sync(0xffffffffu, cs[b], 16);
        }
        if (lane < 8) {
#pragma unroll
          for (int b = 0; b < W; ++b) corr[par][(warp * 16 + b) * 8 + lane] = cs[b];
        }
      } else {
        float c = 0.f;
        if (SRC != kPlain && cj < cur.rows && cb < B) {
          const uint64_t rowbase = uint64_t(cur.r0 + cj) * uint64_t(d.K);
          const uint16_t* xb = p.x[cur.ti] + int64_t(cb) * d.K;
          uint32_t e = ce0 + cq;
          if (kFirst && e < ce1) {
            // the first one was requested while the unit streamed
            if (!f_ready) fetch_first();
            c = fmaf(__uint_as_float(f_x << 16),
                     esc_delta<SRC == kBytesplit ? WCOMP_BYTESPLIT : WCOMP_K15>(f_val, f_lo), c);
            e += cP;
          }
          // four escapes at a time: their loads are independent of each other
          for (; e + 3 * cP < ce1; e += 4 * cP) {
            uint32_t pos[4], val[4], lo[4], xv[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              pos[v] = d.esc_pos[e + v * cP];
              val[v] = load_esc_val(d, e + v * cP);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              lo[v] = SRC == kBytesplit ? uint32_t(d.raw[pos[v]]) : 0u;
              xv[v] = uint32_t(xb[int64_t(uint64_t(pos[v]) - rowbase)]);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
              c = fmaf(__uint_as_float(xv[v] << 16),
                       esc_delta<SRC == kBytesplit ? WCOMP_BYTESPLIT : WCOMP_K15>(val[v], lo[v]), c);
          }
          for (; e < ce1; e += cP) {
            const uint32_t pos = d.esc_pos[e];
            const uint32_t lo = SRC == kBytesplit ? uint32_t(d.raw[pos]) : 0u;
            c = fmaf(__uint_as_float(uint32_t(xb[int64_t(uint64_t(pos) - rowbase)]) << 16),
                     esc_delta<SRC == kBytesplit ? WCOMP_BYTESPLIT : WCOMP_K15>(load_esc_val(d, e), lo), c);
          }
        }
        corr[par][threadIdx.x] = c;
      }
      // the unit after next (requested when this unit started), published
      // with this unit's partial sums
      if (threadIdx.x == 0) next_unit[par] = grabbed;
      __syncthreads();
      if (threadIdx.x < 8 * B && int(threadIdx.x & 7) < cur.rows) {
        const int j = threadIdx.x & 7, bb = threadIdx.x >> 3;
        const int src_lane = (bb & 7) * 4 + (j >> 1), reg = (bb >> 3) * 2 + (j & 1);
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < kMmaWarps; ++w) y += part[par][w][src_lane][reg];
        if (XT) {
#pragma unroll
          for (int w = 0; w < kMmaWarps; ++w) y += corr[par][(w * 16 + bb) * 8 + j];
        } else {
          for (int q = 0; q < cP; ++q) y += corr[par][(q * cbp + bb) * 8 + j];
        }
        p.y[cur.ti][int64_t(bb) * d.N + cur.r0 + j] = y;
      }
    };
    auto step = [&](ChunkBuf& cbuf, ChunkBuf& lbuf) -> bool {
      // request the item after (cur, kb), then compute (cur, kb)
      const bool last = kb + 1 >= cur.kb1;
      if (!last) load_kblock<SRC>(p, cur, kb + 1, g, t, lbuf);
      else if (have_next) {
        MmaUnit first = nxt;
        mma_unit_range(p, warp, first);
        if (first.kb0 < first.kb1) load_kblock<SRC>(p, first, first.kb0, g, t, lbuf);
      }
      if (kb < cur.kb1) {
        const TensorDesc& d = p.d[cur.ti];
        mma_kblock<SRC, XB>(d.t, p.x[cur.ti], d.K, B, cur, kb, lane, cbuf, acc);
      }
      if (kFirst && ++steps_in_unit == 2 && !f_ready) fetch_first();
      if (!last) {
        ++kb;
        return true;
      }
      unit_end();
      if (!have_next) return false;
      cur = nxt;
      mma_unit_range(p, warp, cur);
      ce0 = ne0;
      ce1 = ne1;
      kb = cur.kb0;
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      request_first();
      u_next = next_unit[par];
      par ^= 1;
      if (threadIdx.x == 0) grabbed = atomicAdd(slot, 1u);
      have_next = u_next < total_units;
      if (have_next) {
        mma_unit(p, u_next, cur.ti, nxt);
        row_escapes(nxt, ne0, ne1);
      }
      return true;
    };
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    while (step(b0, b1) && step(b1, b0)) {
    }
  }
  // The last CTA to finish returns the counter slot to zero for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(slot + 1, 1u) == gridDim.x - 1) {
      atomicExch(slot, 0u);
      atomicExch(slot + 1, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Element path (any K, any alignment): one warp per row, static schedule.
// ---------------------------------------------------------------------------
template <int SRC, int BT>
__global__ void __launch_bounds__(kThreads) gemv_generic_kernel(const __grid_constant__ GemvBatch p,
                                                                uint32_t total_rows, int B) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp_id = blockIdx.x * kWarps + (threadIdx.x >> 5);
  for (uint32_t row = warp_id; row < total_rows; row += gridDim.x * kWarps) {
    const int ti = owner(p.set_prefix, p.count, row);
    const TensorDesc& d = p.d[ti];
    const uint16_t* __restrict__ x = p.x[ti];
    const int64_t r = int64_t(row - p.set_prefix[ti]);
    float s[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) s[b] = 0.f;
    for (int64_t k = lane; k < d.K; k += 32) {
      const uint64_t i = uint64_t(r * d.K + k);
      const uint32_t wb = SRC == kPlain ? uint32_t(reinterpret_cast<const uint16_t*>(d.raw)[i])
                                        : decode_elem_placeholder(d, i);
      const float w = __uint_as_float(wb << 16);
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (b < B) s[b] = fmaf(w, __uint_as_float(uint32_t(x[int64_t(b) * d.K + k]) << 16), s[b]);
    }
    if (SRC != kPlain) {
      const uint32_t e0 = d.row_index[r], e1 = d.row_index[r + 1];
      for (uint32_t e = e0 + lane; e < e1; e += 32)
        add_escape<BT>(d, x, B, uint64_t(r) * uint64_t(d.K), d.esc_pos[e], load_esc_val(d, e), s);
    }
    warp_reduce_store<BT>(s, B, p.y[ti], d.N, r, lane);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
int pow2_batch(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

// Per-device scratch: kSlots work-counter pairs, zeroed once at allocation.
// Each launch takes the next slot; its last warp zeroes the slot again.
std::mutex g_scratch_mu;
uint32_t* g_scratch[64] = {nullptr};
std::atomic<uint32_t> g_slot_rr{0};

// The word after the slots is the device error word (bit 0: a staged copy
// never completed).
int scratch(int dev, uint32_t** base) {
  if (dev < 0 || dev >= 64) return WCOMP_EUNSUPPORTED;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch[dev]) {
    uint32_t* p = nullptr;
    const size_t bytes = (kSlots * 2 + 32) * sizeof(uint32_t);
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&p), bytes);
    if (e == cudaSuccess) e = cudaMemset(p, 0, bytes);
    if (e != cudaSuccess) return map_cuda(e);
    g_scratch[dev] = p;
  }
  *base = g_scratch[dev];
  return WCOMP_OK;
}

int counter_slot(int dev, uint32_t** slot) {
  uint32_t* base = nullptr;
  const int st = scratch(dev, &base);
  if (st != WCOMP_OK) return st;
  *slot = base + 2 * (g_slot_rr.fetch_add(1, std::memory_order_relaxed) % kSlots);
  return WCOMP_OK;
}

template <int SRC, int BT, int R, int MINB,
          int MODE = (BT == 1 ? WCOMP_GEMV_MODE1 : BT <= WCOMP_GEMV_MIXED_MAX_B ? 1 : 0),
          int ESC = esc_mode(SRC, BT)>
int launch_vec(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  uint32_t units = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = units;
    units += uint32_t(cdiv(uint64_t(Ns[j]), R));
  }
  b.set_prefix[b.count] = units;
  uint32_t* slot = nullptr;
  int st = counter_slot(dev, &slot);
  if (st != WCOMP_OK) return st;
  // resident CTAs per SM, asked once per instantiation (every thread computes the same value)
  static std::atomic<int> per_sm_cache{0};
  int per_sm = per_sm_cache.load(std::memory_order_relaxed);
  if (!per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<SRC, BT, R, MINB, MODE, ESC>, kThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
      per_sm = 1;
    per_sm_cache.store(per_sm, std::memory_order_relaxed);
  }
  const int blocks = per_sm * sms;
  gemv_kernel<SRC, BT, R, MINB, MODE, ESC><<<blocks, kThreads, 0, s>>>(b, units, B, slot);
  count_launches(1);
  return map_cuda(cudaGetLastError());
}



constexpr uint32_t kStageBudget = 8800;  // shared-memory bytes of staged chunks per warp

template <int SRC, int R>
constexpr int stages() {
  constexpr uint32_t st = (R * Geom<SRC>::row_bytes + 127) & ~127u;
  return kStageBudget / st < 2 ? 2 : int(kStageBudget / st);
}

template <int SRC, int BT, int R, int MINB, int MODE = (BT <= WCOMP_GEMV_MIXED_MAX_B ? 1 : 0)>
int launch_tma(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  constexpr int S = stages<SRC, R>();
  constexpr uint32_t kStage = (R * Geom<SRC>::row_bytes + 127) & ~127u;
  constexpr size_t smem = size_t(kWarps) * (S * kStage + S * 8 + 2 * S * 4);
  uint32_t units = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = units;
    units += uint32_t(cdiv(uint64_t(Ns[j]), R));
  }
  b.set_prefix[b.count] = units;
  uint32_t* base = nullptr;
  int st = scratch(dev, &base);
  if (st != WCOMP_OK) return st;
  uint32_t* slot = nullptr;
  if ((st = counter_slot(dev, &slot)) != WCOMP_OK) return st;
  auto kern = gemv_tma_kernel<SRC, BT, R, MODE, S, MINB>;
  // the shared-memory limit is an attribute of the function in the current device's context
  cudaError_t ae = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ae != cudaSuccess) return map_cuda(ae);
  static std::atomic<int> per_sm_cache{0};
  int per_sm = per_sm_cache.load(std::memory_order_relaxed);
  if (!per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm <= 0)
      per_sm = 1;
    per_sm_cache.store(per_sm, std::memory_order_relaxed);
  }
  kern<<<per_sm * sms, kThreads, smem, s>>>(b, units, B, slot, base + 2 * kSlots);
  count_launches(1);
  return map_cuda(cudaGetLastError());
}

#ifndef WCOMP_GEMV_XT
#define WCOMP_GEMV_XT 1  // K15's escape corrections read a transposed copy of x
#endif
#ifndef WCOMP_GEMV_XT_MIN_B
#define WCOMP_GEMV_XT_MIN_B 3
#endif

// With the transposed x a thread reads all batch rows of an escape's column
// at once (the copy is as wide as the batch: 4, 8 or 16 values per column):
// K15 (escape rate 1.7-3 %) gains from B = 3 (dense-layer set: B = 4 128 ->
// 121.5 us, B = 8 164 -> 131 us, B = 16 251 -> 167 us); at B = 2 the extra
// launch and copy cost more than they save (112 -> 116.5 us), and
// byte-split's few escapes gain nothing.
template <int SRC, int XB, int MINB, int XW>
int launch_mma_xt(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  constexpr bool kXt = XW > 0;
  uint32_t units = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = units;
    units += uint32_t(cdiv(uint64_t(Ns[j]), 8));
  }
  b.set_prefix[b.count] = units;
  uint32_t* slot = nullptr;
  int st = counter_slot(dev, &slot);
  if (st != WCOMP_OK) return st;
  auto kern = gemv_mma_kernel<SRC, XB, MINB, XW>;
  static std::atomic<int> per_sm_cache{0};
  int per_sm = per_sm_cache.load(std::memory_order_relaxed);
  if (!per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMmaThreads, 0) != cudaSuccess || per_sm <= 0)
      per_sm = 1;
    per_sm_cache.store(per_sm, std::memory_order_relaxed);
  }
  XtBatch xt;
  memset(&xt, 0, sizeof(xt));
  uint16_t* xt_mem = nullptr;
  if (kXt) {
    // x transposed into pool memory (freed in stream order after the GEMV)
    uint64_t cols = 0;
    for (int j = 0; j < b.count; ++j) {
      xt.kprefix[j] = uint32_t(cols);
      cols += uint64_t(b.d[j].K);
    }
    if (cols >= (uint64_t(1) << 32)) return WCOMP_EUNSUPPORTED;
    xt.kprefix[b.count] = uint32_t(cols);
    xt.count = b.count;
    cudaError_t e = pool_alloc(reinterpret_cast<void**>(&xt_mem), cols * (kXt ? XW : 1) * sizeof(uint16_t), s);
    if (e != cudaSuccess) return map_cuda(e);
    for (int j = 0; j < b.count; ++j) xt.p[j] = xt_mem + uint64_t(xt.kprefix[j]) * (kXt ? XW : 1);
    const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(cols, 256), uint64_t(sms) * 8));
    transpose_x_kernel<kXt ? XW : 2><<<blocks, 256, 0, s>>>(b, xt, B);
    count_launches(1);
  }
  kern<<<per_sm * sms, kMmaThreads, 0, s>>>(b, units, B, slot, xt);
  count_launches(1);
  const cudaError_t e = cudaGetLastError();
  if (xt_mem) cudaFreeAsync(xt_mem, s);
  return map_cuda(e);
}

template <int SRC, int XB, int MINB>
int launch_mma(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  if (SRC == kK15 && WCOMP_GEMV_XT && B >= WCOMP_GEMV_XT_MIN_B) {
    if (B <= 2) return launch_mma_xt<SRC, XB, MINB, 2>(b, Ns, B, dev, sms, s);
    if (B <= 4) return launch_mma_xt<SRC, XB, MINB, 4>(b, Ns, B, dev, sms, s);
    return launch_mma_xt<SRC, XB, MINB, XB>(b, Ns, B, dev, sms, s);
  }
  return launch_mma_xt<SRC, XB, MINB, 0>(b, Ns, B, dev, sms, s);
}

// Batches from this size up take the tensor-core kernel (measured on the
// dense-layer set): the plain GEMV at every B (its wide per-lane loads and
// x read by a quarter of the lanes beat the FMA kernel even at B = 1), K15
// from B = 2, byte-split from B = 4 (its decode is cheap enough that the FMA
// kernel keeps B = 1..3).  WCOMP_GEMV_MMA_MIN_B overrides all.
#ifndef WCOMP_GEMV_MMA_MIN_B
#define WCOMP_GEMV_MMA_MIN_B 0
#endif
#ifndef WCOMP_GEMV_MMA_MINB
#define WCOMP_GEMV_MMA_MINB 3
#endif
constexpr int mma_min_batch(int src) {
  return WCOMP_GEMV_MMA_MIN_B > 0 ? WCOMP_GEMV_MMA_MIN_B : src == kBytesplit ? 4 : src == kK15 ? 2 : 1;
}

// Rows per unit and CTAs per SM for each batch size (build-time tunables).
#ifndef WCOMP_GEMV_R1
#define WCOMP_GEMV_R1 1
#endif
#ifndef WCOMP_GEMV_R2
#define WCOMP_GEMV_R2 1
#endif
#ifndef WCOMP_GEMV_R4
#define WCOMP_GEMV_R4 2
#endif
#ifndef WCOMP_GEMV_R8
#define WCOMP_GEMV_R8 2
#endif
#ifndef WCOMP_GEMV_R16
#define WCOMP_GEMV_R16 1
#endif

template <int SRC>
int dispatch_vec(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  if (WCOMP_GEMV_TMA) {
    switch (pow2_batch(B)) {
      case 1: return launch_tma<SRC, 1, 1, 3>(b, Ns, B, dev, sms, s);
      case 2: return launch_tma<SRC, 2, WCOMP_GEMV_R2, 3>(b, Ns, B, dev, sms, s);
      case 4: return launch_tma<SRC, 4, WCOMP_GEMV_R4, SRC == kK15 ? 2 : 3>(b, Ns, B, dev, sms, s);
      case 8: return launch_tma<SRC, 8, WCOMP_GEMV_R8, 1>(b, Ns, B, dev, sms, s);
      default: return launch_tma<SRC, 16, WCOMP_GEMV_R16, 1>(b, Ns, B, dev, sms, s);
    }
  }
  if (B >= mma_min_batch(SRC)) {
    if (B <= 8) return launch_mma<SRC, 8, WCOMP_GEMV_MMA_MINB>(b, Ns, B, dev, sms, s);
    return launch_mma<SRC, 16, WCOMP_GEMV_MMA_MINB>(b, Ns, B, dev, sms, s);
  }
  switch (pow2_batch(B)) {
    case 1: return launch_vec<SRC, 1, WCOMP_GEMV_R1, SRC == kK15 ? WCOMP_GEMV_MINB1_K15 : WCOMP_GEMV_MINB1>(b, Ns, B, dev, sms, s);
    case 2: return launch_vec<SRC, 2, WCOMP_GEMV_R2, 3>(b, Ns, B, dev, sms, s);
    case 4: return launch_vec<SRC, 4, WCOMP_GEMV_R4, 2>(b, Ns, B, dev, sms, s);
    case 8: return launch_vec<SRC, 8, WCOMP_GEMV_R8, 1>(b, Ns, B, dev, sms, s);
    default: return launch_vec<SRC, 16, WCOMP_GEMV_R16, 1>(b, Ns, B, dev, sms, s);
  }
}

template <int SRC>
int dispatch_generic(GemvBatch& b, const int64_t* Ns, int B, int sms, cudaStream_t s) {
  uint32_t rows = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = rows;
    rows += uint32_t(Ns[j]);
  }
  b.set_prefix[b.count] = rows;
  const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(rows, kWarps), uint64_t(sms) * 8));
  switch (pow2_batch(B)) {
    case 1: gemv_generic_kernel<SRC, 1><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 2: gemv_generic_kernel<SRC, 2><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 4: gemv_generic_kernel<SRC, 4><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 8: gemv_generic_kernel<SRC, 8><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    default: gemv_generic_kernel<SRC, 16><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
  }
  count_launches(1);
  return map_cuda(cudaGetLastError());
}

// One tensor of a launch request.
struct Item {
  TensorDesc d;
  const uint16_t* x;
  float* y;
  int kind;  // Src for the vector path, 3 + Src for the element path
};

int run_items(Item* items, int count, int B, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = sm_count(dev);
  // longest rows first: the tail of the dynamic schedule is made of short units
  std::stable_sort(items, items + count, [](const Item& a, const Item& b) { return a.d.K > b.d.K; });
  for (int kind = 0; kind < 6; ++kind) {
    GemvBatch bt;
    memset(&bt, 0, sizeof(bt));
    int64_t Ns[kMaxBatch];
    auto flush = [&]() -> int {
      if (!bt.count) return WCOMP_OK;
      int st;
      switch (kind) {
        case 0: st = dispatch_vec<kBytesplit>(bt, Ns, B, dev, sms, s); break;
        case 1: st = dispatch_vec<kK15>(bt, Ns, B, dev, sms, s); break;
        case 2: st = dispatch_vec<kPlain>(bt, Ns, B, dev, sms, s); break;
        case 3: st = dispatch_generic<kBytesplit>(bt, Ns, B, sms, s); break;
        case 4: st = dispatch_generic<kK15>(bt, Ns, B, sms, s); break;
        default: st = dispatch_generic<kPlain>(bt, Ns, B, sms, s); break;
      }
      memset(&bt, 0, sizeof(bt));
      return st;
    };
    for (int i = 0; i < count; ++i) {
      if (items[i].kind != kind) continue;
      bt.d[bt.count] = items[i].d;
      bt.x[bt.count] = items[i].x;
      bt.y[bt.count] = items[i].y;
      Ns[bt.count] = items[i].d.N;
      if (++bt.count == kMaxBatch) {
        const int st = flush();
        if (st != WCOMP_OK) return st;
      }
    }
    const int st = flush();
    if (st != WCOMP_OK) return st;
  }
  return WCOMP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; }

int gemv_containers(const wcomp_container* const* cs, const uint16_t* const* xs, int B, float* const* ys, int count,
                    cudaStream_t s) {
  if (B < 1 || B > 16) return WCOMP_EINVAL;
  std::vector<Item> items(count);
  for (int i = 0; i < count; ++i) {
    if (!cs[i] || !xs[i] || !ys[i]) return WCOMP_EINVAL;
    if (cs[i]->L.N >= (int64_t(1) << 31)) return WCOMP_EUNSUPPORTED;
    items[i].d = make_desc(cs[i]);
    items[i].x = xs[i];
    items[i].y = ys[i];
    const bool vec = cs[i]->L.K % kGroup == 0 && aligned16(xs[i]) && aligned32(cs[i]->d_main);
    items[i].kind = (vec ? 0 : 3) + cs[i]->L.scheme;
  }
  return run_items(items.data(), count, B, s);
}

int gemv_plain(const uint16_t* const* ws, const int64_t* Ns, const int64_t* Ks, const uint16_t* const* xs, int B,
               float* const* ys, int count, cudaStream_t s) {
  if (B < 1 || B > 16) return WCOMP_EINVAL;
  std::vector<Item> items(count);
  for (int i = 0; i < count; ++i) {
    if (!ws[i] || !xs[i] || !ys[i] || Ns[i] <= 0 || Ks[i] <= 0) return WCOMP_EINVAL;
    if (Ns[i] >= (int64_t(1) << 31)) return WCOMP_EUNSUPPORTED;
    TensorDesc d{};
    d.raw = reinterpret_cast<const uint8_t*>(ws[i]);
    d.N = Ns[i];
    d.K = Ks[i];
    d.n = uint64_t(Ns[i]) * uint64_t(Ks[i]);
    d.scheme = kPlain;
    items[i].d = d;
    items[i].x = xs[i];
    items[i].y = ys[i];
    const bool vec = Ks[i] % kGroup == 0 && aligned16(xs[i]) && aligned32(ws[i]);
    items[i].kind = vec ? kPlain : 3 + kPlain;
  }
  return run_items(items.data(), count, B, s);
}

}  // namespace
}  // namespace wc

using namespace wc;

extern "C" int wcomp_device_check(void* stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  uint32_t* base = nullptr;
  int st = scratch(dev, &base);
  if (st != WCOMP_OK) return st;
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, base + 2 * kSlots, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return map_cuda(e);
  if (word) {
    cudaMemsetAsync(base + 2 * kSlots, 0, sizeof(uint32_t), s);
    cudaStreamSynchronize(s);
    return WCOMP_ETIMEOUT;
  }
  return WCOMP_OK;
}

extern "C" int wcomp_gemv(const wcomp_container* c, const uint16_t* d_x, int B, float* d_y, void* stream) {
  if (!c || !d_x || !d_y) return WCOMP_EINVAL;
  return gemv_containers(&c, &d_x, B, &d_y, 1, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_gemv_batched(const wcomp_container* const* containers, const uint16_t* const* d_x, int B,
                                  float* const* d_y, int count, void* stream) {
  if (!containers || !d_x || !d_y || count <= 0) return WCOMP_EINVAL;
  return gemv_containers(containers, d_x, B, d_y, count, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_gemv_bf16(const uint16_t* d_w, int64_t N, int64_t K, const uint16_t* d_x, int B, float* d_y,
                               void* stream) {
  if (!d_w || !d_x || !d_y || N <= 0 || K <= 0) return WCOMP_EINVAL;
  return gemv_plain(&d_w, &N, &K, &d_x, B, &d_y, 1, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_gemv_bf16_batched(const uint16_t* const* d_w, const int64_t* N, const int64_t* K,
                                       const uint16_t* const* d_x, int B, float* const* d_y, int count, void* stream) {
  if (!d_w || !N || !K || !d_x || !d_y || count <= 0) return WCOMP_EINVAL;
  return gemv_plain(d_w, N, K, d_x, B, d_y, count, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Fused GEMV that allocates nothing.
//
// wcomp_gemv takes its work counters from a device buffer that the library
// allocates with cudaMalloc on first use.  Some callers cannot let a library
// allocate device memory: a serving loop that fixed its memory budget up
// front, or code that must not meet the implicit device synchronisation that
// a first cudaMalloc (or any cudaFree) can bring.  wcomp_gemv_noalloc runs the
// same kernel with its counters in the static device array below instead.
// The array is part of the library image, so every GPU that loads the library
// keeps it until the process exits.  Every call shares it.
// ---------------------------------------------------------------------------
namespace wc {
namespace {

constexpr int kNoAllocWords = 64;  // 256 bytes: [0] work counter, [1] completion counter, rest unused
// A call may cover at most this many rows: the work counter runs past the
// row count by one grab per warp of the grid and must stay within 32 bits.
constexpr int64_t kNoAllocMaxRows = (int64_t(1) << 31) - (int64_t(1) << 20);

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

std::mutex g_noalloc_mu;
uint32_t* g_noalloc_ptr[64] = {nullptr};

// Device address of the static array on device `dev` (which must be current).
// The host-side name of the array is not a device address; the runtime gives
// the real one, looked up once per device.
int noalloc_scratch(int dev, uint32_t** out) {
  if (dev < 0 || dev >= 64) return WCOMP_EUNSUPPORTED;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return map_cuda(e);
    g_noalloc_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return WCOMP_OK;
}

template <int SRC, int BT, int R, int MINB,
          int MODE = (BT == 1 ? WCOMP_GEMV_MODE1 : BT <= WCOMP_GEMV_MIXED_MAX_B ? 1 : 0)>
int launch_vec_on(GemvBatch& b, int64_t N, int B, int sms, uint32_t* slot, cudaStream_t s) {
  b.set_prefix[0] = 0;
  const uint32_t units = uint32_t(cdiv(uint64_t(N), R));
  b.set_prefix[1] = units;
  auto kern = gemv_kernel<SRC, BT, R, MINB, MODE, esc_mode(SRC, BT)>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess || per_sm <= 0)
    per_sm = 1;
  kern<<<per_sm * sms, kThreads, 0, s>>>(b, units, B, slot);
  count_launches(1);
  return map_cuda(cudaGetLastError());
}

template <int SRC, int XB>
int launch_mma_on(GemvBatch& b, int64_t N, int B, int sms, uint32_t* slot, cudaStream_t s) {
  b.set_prefix[0] = 0;
  const uint32_t units = uint32_t(cdiv(uint64_t(N), 8));
  b.set_prefix[1] = units;
  auto kern = gemv_mma_kernel<SRC, XB, WCOMP_GEMV_MMA_MINB>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMmaThreads, 0) != cudaSuccess || per_sm <= 0)
    per_sm = 1;
  XtBatch xt;
  memset(&xt, 0, sizeof(xt));
  kern<<<per_sm * sms, kMmaThreads, 0, s>>>(b, units, B, slot, xt);
  count_launches(1);
  return map_cuda(cudaGetLastError());
}

template <int SRC>
int dispatch_vec_on(GemvBatch& b, int64_t N, int B, int sms, uint32_t* slot, cudaStream_t s) {
  if (B >= mma_min_batch(SRC))
    return B <= 8 ? launch_mma_on<SRC, 8>(b, N, B, sms, slot, s) : launch_mma_on<SRC, 16>(b, N, B, sms, slot, s);
  switch (pow2_batch(B)) {
    case 1: return launch_vec_on<SRC, 1, WCOMP_GEMV_R1, SRC == kK15 ? WCOMP_GEMV_MINB1_K15 : WCOMP_GEMV_MINB1>(
        b, N, B, sms, slot, s);
    case 2: return launch_vec_on<SRC, 2, WCOMP_GEMV_R2, 3>(b, N, B, sms, slot, s);
    case 4: return launch_vec_on<SRC, 4, WCOMP_GEMV_R4, 2>(b, N, B, sms, slot, s);
    case 8: return launch_vec_on<SRC, 8, WCOMP_GEMV_R8, 1>(b, N, B, sms, slot, s);
    default: return launch_vec_on<SRC, 16, WCOMP_GEMV_R16, 1>(b, N, B, sms, slot, s);
  }
}

}  // namespace
}  // namespace wc

extern "C" int wcomp_gemv_noalloc(const wcomp_container* c, const uint16_t* d_x, int B, float* d_y, void* stream) {
  if (!c || !d_x || !d_y || B < 1 || B > 16) return WCOMP_EINVAL;
  if (c->L.N > kNoAllocMaxRows) return WCOMP_EUNSUPPORTED;
  int dev = 0;
  cudaGetDevice(&dev);
  uint32_t* scratch = nullptr;
  int st = noalloc_scratch(dev, &scratch);
  if (st != WCOMP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The counters must start at zero; a memset allocates nothing.
  cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return map_cuda(e);
  const int sms = sm_count(dev);
  GemvBatch b;
  memset(&b, 0, sizeof(b));
  b.count = 1;
  b.d[0] = make_desc(c);
  b.x[0] = d_x;
  b.y[0] = d_y;
  const int64_t N = c->L.N;
  const bool vec = c->L.K % kGroup == 0 && aligned16(d_x) && aligned32(c->d_main);
  if (!vec) {
    // the element path uses no scratch at all
    return c->L.scheme == WCOMP_BYTESPLIT ? dispatch_generic<kBytesplit>(b, &N, B, sms, s)
                                          : dispatch_generic<kK15>(b, &N, B, sms, s);
  }
  return c->L.scheme == WCOMP_BYTESPLIT ? dispatch_vec_on<kBytesplit>(b, N, B, sms, scratch, s)
                                        : dispatch_vec_on<kK15>(b, N, B, sms, scratch, s);
}
