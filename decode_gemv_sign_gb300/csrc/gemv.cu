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
// Work decomposition.  A unit of work is a set of R consecutive rows of one
// tensor; a launch covers the units of every tensor in the batch.  The grid is
// persistent (as many CTAs as fit on the GPU at once) and every warp grabs
// units from a global counter, one at a time, so the GPU drains evenly even
// when the tensors differ in shape.  Inside a unit the warp walks the rows:
// lane l takes the 32-element groups l, l+32, ..., keeps the next group's
// loads in flight while it computes the current one (register double
// buffering), loads each stream with vector loads that bypass L1, rebuilds
// BF16 pairs with prmt lookups, widens them to fp32 with a shift / mask and
// accumulates in fp32 (mixed-precision or packed fp32x2 FMAs, see below).  x is read through L1, where it stays
// (every warp of the SM reads the same x).
//
// Escapes.  An escaped weight decodes to the placeholder (symbol 0, so
// |w| < 2^-125).  Each lane adds x * (w_true - w_placeholder) for a share of
// the unit's escapes, found in O(1) through the row index; their positions
// and values are requested before the main loop so the loads overlap it.
// Lanes are combined with a fixed butterfly: results do not depend on which
// warp ran which unit.
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

// FMA forms.  MODE 0 widens weights and x to fp32 and issues packed fp32x2
// FMAs (x is widened once per unit of R rows).  MODE 1 feeds the BF16 halves
// of the pair words straight into mixed-precision FMAs (bf16 x bf16 + fp32);
// the product of two BF16 values is exact in fp32, so both forms round the
// same sums.  MODE 1 saves the widening work and wins for small batches.
#ifndef WCOMP_GEMV_MIXED_MAX_B
#define WCOMP_GEMV_MIXED_MAX_B 2
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

// Find the tensor that owns global unit `u`.
__device__ __forceinline__ int owner(const uint32_t* prefix, int count, uint32_t u) {
  int i = 0;
  while (i + 1 < count && prefix[i + 1] <= u) ++i;
  return i;
}

// ---------------------------------------------------------------------------
// Weight sources: one 32-element group of one row.
// ---------------------------------------------------------------------------
struct GroupBuf {
  uint32_t v[16];
};

template <int SRC>
__device__ __forceinline__ void load_buf(const TensorDesc& d, uint64_t g, GroupBuf& b) {
  if (SRC == kBytesplit) {
    const uint4 c = ld_stream_v4(d.codes + 16 * g);
    b.v[0] = c.x; b.v[1] = c.y; b.v[2] = c.z; b.v[3] = c.w;
    uint32_t r[8];
    ld_stream_v8(d.raw + 32 * g, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) b.v[4 + i] = r[i];
  } else if (SRC == kK15) {
    const uint4 c = ld_stream_v4(d.codes + 16 * g);
    const uint4 a = ld_stream_v4(d.pa + 16 * g);
    const uint2 pb = ld_stream_v2(d.pb + 8 * g);
    b.v[0] = c.x; b.v[1] = c.y; b.v[2] = c.z; b.v[3] = c.w;
    b.v[4] = a.x; b.v[5] = a.y; b.v[6] = a.z; b.v[7] = a.w;
    b.v[8] = pb.x; b.v[9] = pb.y;
    b.v[10] = ld_stream_u32(d.pc + 4 * g);
  } else {
    uint32_t r[8];
    const uint8_t* w = d.raw + 64 * g;
    ld_stream_v8(w, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) b.v[i] = r[i];
    ld_stream_v8(w + 32, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) b.v[8 + i] = r[i];
  }
}

// BF16 pairs of code word I (elements 8I .. 8I+7) of a loaded group.
template <int SRC, int I>
__device__ __forceinline__ void pairs8(const RegTable& t, const GroupBuf& b, uint32_t (&w)[4]) {
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
    const uint32_t a[4] = {b.v[4], b.v[5], b.v[6], b.v[7]};
    const uint32_t pb[2] = {b.v[8], b.v[9]};
    uint32_t e0, e1;
    lookup8(t.e0, m7, m, e0, e1);
    l0 = k15_mant<2 * I>(a, pb, b.v[10]) | e0;
    l1 = k15_mant<2 * I + 1>(a, pb, b.v[10]) | e1;
  }
  w[0] = prmt(l0, h0, 0x5140);
  w[1] = prmt(l0, h0, 0x7362);
  w[2] = prmt(l1, h1, 0x5140);
  w[3] = prmt(l1, h1, 0x7362);
}

template <int SRC, int BT, int R, int MODE>
__device__ __forceinline__ void compute_group(const TensorDesc& d, const uint16_t* __restrict__ xg, int64_t K, int B,
                                              const GroupBuf (&buf)[R], const bool (&live)[R],
                                              float2 (&acc)[R][BT]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t xw[BT][4];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      if (b < B) {
        const uint4 v = ld_x_v4(xg + int64_t(b) * K + 8 * i);
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
      if (i == 0) pairs8<SRC, 0>(d.t, buf[j], w);
      else if (i == 1) pairs8<SRC, 1>(d.t, buf[j], w);
      else if (i == 2) pairs8<SRC, 2>(d.t, buf[j], w);
      else pairs8<SRC, 3>(d.t, buf[j], w);
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
template <int SRC, int BT, int R, int MINB, int MODE>
__global__ void __launch_bounds__(kThreads, MINB)
    gemv_kernel(const __grid_constant__ GemvBatch p, uint32_t total_units, int B, uint32_t* __restrict__ slot) {
  const int lane = threadIdx.x & 31;
  uint32_t u = grab(slot, lane);
  while (u < total_units) {
    const uint32_t u_next = grab(slot, lane);  // in flight while this unit runs
    const int ti = owner(p.set_prefix, p.count, u);
    const TensorDesc& d = p.d[ti];
    const uint16_t* __restrict__ x = p.x[ti];
    const int64_t r0 = int64_t(u - p.set_prefix[ti]) * R;
    const int64_t K = d.K;
    const uint64_t KG = uint64_t(K) / kGroup;
    bool live[R];
#pragma unroll
    for (int j = 0; j < R; ++j) live[j] = r0 + j < d.N;
    float2 acc[R][BT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[j][b] = make_float2(0.f, 0.f);

    GroupBuf b0[R], b1[R];
    uint64_t gk = lane;
    if (gk < KG) {
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (live[j]) load_buf<SRC>(d, uint64_t(r0 + j) * KG + gk, b0[j]);
    }
    // escape slice of the unit: index now, first entries right after
    uint32_t e_lo = 0, e_hi = 0, p0 = 0, v0 = 0;
    if (SRC != kPlain) {
      const int64_t r_end = r0 + R < d.N ? r0 + R : d.N;
      e_lo = d.row_index[r0];
      e_hi = d.row_index[r_end];
      if (e_lo + lane < e_hi) {
        p0 = d.esc_pos[e_lo + lane];
        v0 = load_esc_val(d, e_lo + lane);
      }
    }
    for (; gk < KG; gk += 64) {
      const bool more = gk + 32 < KG;
      if (more) {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (live[j]) load_buf<SRC>(d, uint64_t(r0 + j) * KG + gk + 32, b1[j]);
      }
      compute_group<SRC, BT, R, MODE>(d, x + gk * kGroup, K, B, b0, live, acc);
      if (!more) break;
      if (gk + 64 < KG) {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (live[j]) load_buf<SRC>(d, uint64_t(r0 + j) * KG + gk + 64, b0[j]);
      }
      compute_group<SRC, BT, R, MODE>(d, x + (gk + 32) * kGroup, K, B, b1, live, acc);
    }

    float s[R][BT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int b = 0; b < BT; ++b) s[j][b] = acc[j][b].x + acc[j][b].y;
    if (SRC != kPlain) {
      // escapes of the unit, lane-strided; each goes to the row that holds it
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
    u = u_next;
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

int counter_slot(int dev, uint32_t** slot) {
  if (dev < 0 || dev >= 64) return WCOMP_EUNSUPPORTED;
  {
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch[dev]) {
      uint32_t* p = nullptr;
      cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&p), kSlots * 2 * sizeof(uint32_t));
      if (e == cudaSuccess) e = cudaMemset(p, 0, kSlots * 2 * sizeof(uint32_t));
      if (e != cudaSuccess) return map_cuda(e);
      g_scratch[dev] = p;
    }
  }
  *slot = g_scratch[dev] + 2 * (g_slot_rr.fetch_add(1, std::memory_order_relaxed) % kSlots);
  return WCOMP_OK;
}

template <int SRC, int BT, int R, int MINB, int MODE = (BT <= WCOMP_GEMV_MIXED_MAX_B ? 1 : 0)>
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
  static int per_sm_cache = 0;
  if (!per_sm_cache) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<SRC, BT, R, MINB, MODE>, kThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
      per_sm = 1;
    per_sm_cache = per_sm;
  }
  const int blocks = per_sm_cache * sms;
  gemv_kernel<SRC, BT, R, MINB, MODE><<<blocks, kThreads, 0, s>>>(b, units, B, slot);
  count_launches(1);
  return map_cuda(cudaGetLastError());
}

template <int SRC>
int dispatch_vec(GemvBatch& b, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  switch (pow2_batch(B)) {
    case 1: return launch_vec<SRC, 1, 1, 3>(b, Ns, B, dev, sms, s);
    case 2: return launch_vec<SRC, 2, 1, 3>(b, Ns, B, dev, sms, s);
    case 4: return launch_vec<SRC, 4, 2, 2>(b, Ns, B, dev, sms, s);
    case 8: return launch_vec<SRC, 8, 1, 2>(b, Ns, B, dev, sms, s);
    default: return launch_vec<SRC, 16, 1, 1>(b, Ns, B, dev, sms, s);
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
