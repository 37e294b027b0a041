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
// Work decomposition: a warp owns a set of R consecutive rows and walks the
// whole row; lane l takes the 32-element groups l, l+32, ... .  For each group
// the lane loads 16 code bytes and 32 raw bytes (byte-split) or 28 plane bytes
// (K15) per row with streaming vector loads that bypass L1, rebuilds BF16
// pairs with prmt lookups, widens them to fp32 with a shift / mask and
// accumulates with packed fp32x2 FMAs.  x is read through L1 (it is shared by
// every warp of the SM).  Escaped weights decode to the placeholder (symbol
// 0, |w| < 2^-125); each lane then adds x * (w_true - w_placeholder) for a
// share of the row's escapes, found in O(1) through the row index.  Lanes are
// combined with a fixed butterfly, so results do not depend on scheduling.
#include <string.h>

#include <algorithm>

#include "wcomp_impl.cuh"

namespace wc {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct F2 {
  float x, y;
};

__device__ __forceinline__ void fma2(F2& acc, uint32_t w_pair, float x0, float x1) {
  // acc.{x,y} += {w_lo, w_hi} * {x0, x1} as one packed fp32x2 FMA
  const float w0 = bf16_lo(w_pair), w1 = bf16_hi(w_pair);
  uint64_t a, b, c, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(w0), "f"(w1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(c) : "f"(acc.x), "f"(acc.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(d));
}

__device__ __forceinline__ uint4 ld_x_v4(const uint16_t* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Find the tensor that owns global row set `set`.
__device__ __forceinline__ int owner(const uint32_t* prefix, int count, uint32_t set) {
  int i = 0;
  while (i + 1 < count && prefix[i + 1] <= set) ++i;
  return i;
}

// Escape correction for row r: lane-strided share of the row's escapes.
template <int BT>
__device__ __forceinline__ void escape_correction(const TensorDesc& d, const uint16_t* __restrict__ x, int B,
                                                  int64_t r, int lane, float (&s)[BT]) {
  const uint32_t e0 = d.row_index[r], e1 = d.row_index[r + 1];
  for (uint32_t e = e0 + lane; e < e1; e += 32) {
    const uint32_t p = d.esc_pos[e];
    const int64_t k = int64_t(p) - r * d.K;
    const uint32_t wt = escape_word(d, e, p);
    const uint32_t wph = d.scheme == WCOMP_BYTESPLIT ? (wt & 0xFFu) : (wt & 0x7Fu);
    const float delta = __uint_as_float(wt << 16) - __uint_as_float(wph << 16);
#pragma unroll
    for (int b = 0; b < BT; ++b)
      if (b < B) s[b] = fmaf(__uint_as_float(uint32_t(x[int64_t(b) * d.K + k]) << 16), delta, s[b]);
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

// ---------------------------------------------------------------------------
// Fused decode-GEMV, vector path (K % 32 == 0, 16-byte aligned x).
// ---------------------------------------------------------------------------
template <int SCHEME, int BT, int R>
__global__ void __launch_bounds__(kThreads) gemv_fused_kernel(const __grid_constant__ GemvBatch p, uint32_t total_sets,
                                                              int B) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp_id = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * kWarps;
  for (uint32_t set = warp_id; set < total_sets; set += nwarps) {
    const int ti = owner(p.set_prefix, p.count, set);
    const TensorDesc& d = p.d[ti];
    const uint16_t* __restrict__ x = p.x[ti];
    const int64_t r0 = int64_t(set - p.set_prefix[ti]) * R;
    const int64_t K = d.K;
    const uint64_t KG = uint64_t(K) / kGroup;
    F2 acc[R][BT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[j][b] = F2{0.f, 0.f};
    bool live[R];
#pragma unroll
    for (int j = 0; j < R; ++j) live[j] = r0 + j < d.N;

    for (uint64_t gk = lane; gk < KG; gk += 32) {
      uint32_t cw[R][4], rw[R][8];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (live[j]) {
          load_group<SCHEME>(d, uint64_t(r0 + j) * KG + gk, cw[j], rw[j]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) cw[j][i] = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) rw[j][i] = 0;
        }
      }
      const uint16_t* xg = x + gk * kGroup;
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // 8 elements per code word
        float xf[BT][8];
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          if (b < B) {
            const uint4 v = ld_x_v4(xg + int64_t(b) * K + 8 * i);
            xf[b][0] = bf16_lo(v.x); xf[b][1] = bf16_hi(v.x);
            xf[b][2] = bf16_lo(v.y); xf[b][3] = bf16_hi(v.y);
            xf[b][4] = bf16_lo(v.z); xf[b][5] = bf16_hi(v.z);
            xf[b][6] = bf16_lo(v.w); xf[b][7] = bf16_hi(v.w);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) xf[b][k] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const QuadMasks m = code_masks(cw[j][i]);
          const uint32_t m7 = cw[j][i] & 0x77777777u;
          uint32_t h0, h1;
          lookup8(d.t.hi, m7, m, h0, h1);
          uint32_t l0 = rw[j][2 * i], l1 = rw[j][2 * i + 1];
          if (SCHEME == WCOMP_K15) {
            uint32_t e0, e1;
            lookup8(d.t.e0, m7, m, e0, e1);
            l0 |= e0;
            l1 |= e1;
          }
          const uint32_t w01 = prmt(l0, h0, 0x5140), w23 = prmt(l0, h0, 0x7362);
          const uint32_t w45 = prmt(l1, h1, 0x5140), w67 = prmt(l1, h1, 0x7362);
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            fma2(acc[j][b], w01, xf[b][0], xf[b][1]);
            fma2(acc[j][b], w23, xf[b][2], xf[b][3]);
            fma2(acc[j][b], w45, xf[b][4], xf[b][5]);
            fma2(acc[j][b], w67, xf[b][6], xf[b][7]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (!live[j]) continue;  // uniform across the warp
      float s[BT];
#pragma unroll
      for (int b = 0; b < BT; ++b) s[b] = acc[j][b].x + acc[j][b].y;
      escape_correction<BT>(d, x, B, r0 + j, lane, s);
      warp_reduce_store<BT>(s, B, p.y[ti], d.N, r0 + j, lane);
    }
  }
}

// ---------------------------------------------------------------------------
// Fused decode-GEMV, element path (any K, any alignment): one warp per row.
// ---------------------------------------------------------------------------
template <int BT>
__global__ void __launch_bounds__(kThreads) gemv_fused_generic_kernel(const __grid_constant__ GemvBatch p,
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
      const float w = __uint_as_float(decode_elem_placeholder(d, uint64_t(r * d.K + k)) << 16);
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (b < B) s[b] = fmaf(w, __uint_as_float(uint32_t(x[int64_t(b) * d.K + k]) << 16), s[b]);
    }
    escape_correction<BT>(d, x, B, r, lane, s);
    warp_reduce_store<BT>(s, B, p.y[ti], d.N, r, lane);
  }
}

// ---------------------------------------------------------------------------
// Plain BF16 GEMV (the comparison kernel): same decomposition, W read raw.
// ---------------------------------------------------------------------------
struct PlainArgs {
  const uint16_t* w;
  const uint16_t* x;
  float* y;
  int64_t N, K;
};

template <int BT, int R>
__global__ void __launch_bounds__(kThreads) gemv_bf16_kernel(const __grid_constant__ PlainArgs a, int B) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp_id = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * kWarps;
  const int64_t K = a.K;
  const uint64_t KG = uint64_t(K) / kGroup;
  const uint32_t sets = uint32_t(cdiv(uint64_t(a.N), R));
  for (uint32_t set = warp_id; set < sets; set += nwarps) {
    const int64_t r0 = int64_t(set) * R;
    F2 acc[R][BT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[j][b] = F2{0.f, 0.f};
    bool live[R];
#pragma unroll
    for (int j = 0; j < R; ++j) live[j] = r0 + j < a.N;
    for (uint64_t gk = lane; gk < KG; gk += 32) {
      uint32_t wv[R][16];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (live[j]) {
          const uint16_t* src = a.w + (uint64_t(r0 + j) * KG + gk) * kGroup;
          ld_stream_v8(src, *reinterpret_cast<uint32_t(*)[8]>(&wv[j][0]));
          ld_stream_v8(src + 16, *reinterpret_cast<uint32_t(*)[8]>(&wv[j][8]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) wv[j][i] = 0;
        }
      }
      const uint16_t* xg = a.x + gk * kGroup;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float xf[BT][8];
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          if (b < B) {
            const uint4 v = ld_x_v4(xg + int64_t(b) * K + 8 * i);
            xf[b][0] = bf16_lo(v.x); xf[b][1] = bf16_hi(v.x);
            xf[b][2] = bf16_lo(v.y); xf[b][3] = bf16_hi(v.y);
            xf[b][4] = bf16_lo(v.z); xf[b][5] = bf16_hi(v.z);
            xf[b][6] = bf16_lo(v.w); xf[b][7] = bf16_hi(v.w);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) xf[b][k] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            fma2(acc[j][b], wv[j][4 * i + 0], xf[b][0], xf[b][1]);
            fma2(acc[j][b], wv[j][4 * i + 1], xf[b][2], xf[b][3]);
            fma2(acc[j][b], wv[j][4 * i + 2], xf[b][4], xf[b][5]);
            fma2(acc[j][b], wv[j][4 * i + 3], xf[b][6], xf[b][7]);
          }
      }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (!live[j]) continue;
      float s[BT];
#pragma unroll
      for (int b = 0; b < BT; ++b) s[b] = acc[j][b].x + acc[j][b].y;
      warp_reduce_store<BT>(s, B, a.y, a.N, r0 + j, lane);
    }
  }
}

template <int BT>
__global__ void __launch_bounds__(kThreads) gemv_bf16_generic_kernel(const __grid_constant__ PlainArgs a, int B) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp_id = blockIdx.x * kWarps + (threadIdx.x >> 5);
  for (int64_t r = warp_id; r < a.N; r += int64_t(gridDim.x) * kWarps) {
    float s[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) s[b] = 0.f;
    for (int64_t k = lane; k < a.K; k += 32) {
      const float w = __uint_as_float(uint32_t(a.w[r * a.K + k]) << 16);
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (b < B) s[b] = fmaf(w, __uint_as_float(uint32_t(a.x[int64_t(b) * a.K + k]) << 16), s[b]);
    }
    warp_reduce_store<BT>(s, B, a.y, a.N, r, lane);
  }
}

// ---------------------------------------------------------------------------
// Host dispatch.
// ---------------------------------------------------------------------------
int pow2_batch(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

template <int SCHEME, int BT, int R>
void launch_fused(const GemvBatch& b, uint32_t sets, int B, int sms, cudaStream_t s) {
  const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(sets, kWarps), uint64_t(sms) * 8));
  gemv_fused_kernel<SCHEME, BT, R><<<blocks, kThreads, 0, s>>>(b, sets, B);
  count_launches(1);
}

template <int SCHEME>
void dispatch_fused(GemvBatch& b, const int64_t* Ns, int B, int sms, cudaStream_t s) {
  const int BT = pow2_batch(B);
  const int R = BT >= 16 ? 1 : 2;
  uint32_t sets = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = sets;
    sets += uint32_t(cdiv(uint64_t(Ns[j]), R));
  }
  b.set_prefix[b.count] = sets;
  switch (BT) {
    case 1: launch_fused<SCHEME, 1, 2>(b, sets, B, sms, s); break;
    case 2: launch_fused<SCHEME, 2, 2>(b, sets, B, sms, s); break;
    case 4: launch_fused<SCHEME, 4, 2>(b, sets, B, sms, s); break;
    case 8: launch_fused<SCHEME, 8, 2>(b, sets, B, sms, s); break;
    default: launch_fused<SCHEME, 16, 1>(b, sets, B, sms, s); break;
  }
}

void dispatch_generic(GemvBatch& b, const int64_t* Ns, int B, int sms, cudaStream_t s) {
  uint32_t rows = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = rows;
    rows += uint32_t(Ns[j]);
  }
  b.set_prefix[b.count] = rows;
  const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(rows, kWarps), uint64_t(sms) * 8));
  switch (pow2_batch(B)) {
    case 1: gemv_fused_generic_kernel<1><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 2: gemv_fused_generic_kernel<2><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 4: gemv_fused_generic_kernel<4><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    case 8: gemv_fused_generic_kernel<8><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
    default: gemv_fused_generic_kernel<16><<<blocks, kThreads, 0, s>>>(b, rows, B); break;
  }
  count_launches(1);
}

bool fast_ok(const wcomp_container* c, const uint16_t* x) {
  return c->L.K % kGroup == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(c->d_main) & 31) == 0;
}

int launch_gemv(const wcomp_container* const* cs, const uint16_t* const* xs, int B, float* const* ys, int count,
                cudaStream_t s) {
  if (B < 1 || B > 16) return WCOMP_EINVAL;
  for (int i = 0; i < count; ++i) {
    if (!cs[i] || !xs[i] || !ys[i]) return WCOMP_EINVAL;
    if (cs[i]->L.N >= (int64_t(1) << 31)) return WCOMP_EUNSUPPORTED;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = sm_count(dev);
  // Three kinds of launches: vector path per scheme, element path for the rest.
  for (int kind = 0; kind < 3; ++kind) {
    GemvBatch b;
    memset(&b, 0, sizeof(b));
    int64_t Ns[kMaxBatch];
    auto flush = [&]() {
      if (!b.count) return;
      if (kind == 0) dispatch_fused<WCOMP_BYTESPLIT>(b, Ns, B, sms, s);
      else if (kind == 1) dispatch_fused<WCOMP_K15>(b, Ns, B, sms, s);
      else dispatch_generic(b, Ns, B, sms, s);
      memset(&b, 0, sizeof(b));
    };
    for (int i = 0; i < count; ++i) {
      const wcomp_container* c = cs[i];
      const bool fast = fast_ok(c, xs[i]);
      const int k = fast ? c->L.scheme : 2;
      if (k != kind) continue;
      b.d[b.count] = make_desc(c);
      b.x[b.count] = xs[i];
      b.y[b.count] = ys[i];
      Ns[b.count] = c->L.N;
      if (++b.count == kMaxBatch) flush();
    }
    flush();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return map_cuda(e);
  }
  return WCOMP_OK;
}

}  // namespace
}  // namespace wc

using namespace wc;

extern "C" int wcomp_gemv(const wcomp_container* c, const uint16_t* d_x, int B, float* d_y, void* stream) {
  if (!c || !d_x || !d_y) return WCOMP_EINVAL;
  return launch_gemv(&c, &d_x, B, &d_y, 1, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_gemv_batched(const wcomp_container* const* containers, const uint16_t* const* d_x, int B,
                                  float* const* d_y, int count, void* stream) {
  if (!containers || !d_x || !d_y || count <= 0) return WCOMP_EINVAL;
  return launch_gemv(containers, d_x, B, d_y, count, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_gemv_bf16(const uint16_t* d_w, int64_t N, int64_t K, const uint16_t* d_x, int B, float* d_y,
                               void* stream) {
  if (!d_w || !d_x || !d_y || N <= 0 || K <= 0 || B < 1 || B > 16) return WCOMP_EINVAL;
  if (N >= (int64_t(1) << 31)) return WCOMP_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = sm_count(dev);
  PlainArgs a{d_w, d_x, d_y, N, K};
  const bool fast = K % kGroup == 0 && (reinterpret_cast<uintptr_t>(d_w) & 31) == 0 &&
                    (reinterpret_cast<uintptr_t>(d_x) & 15) == 0;
  const int BT = pow2_batch(B);
  if (fast) {
    const int R = BT >= 16 ? 1 : 2;
    const uint32_t sets = uint32_t(cdiv(uint64_t(N), R));
    const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(sets, kWarps), uint64_t(sms) * 8));
    switch (BT) {
      case 1: gemv_bf16_kernel<1, 2><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 2: gemv_bf16_kernel<2, 2><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 4: gemv_bf16_kernel<4, 2><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 8: gemv_bf16_kernel<8, 2><<<blocks, kThreads, 0, s>>>(a, B); break;
      default: gemv_bf16_kernel<16, 1><<<blocks, kThreads, 0, s>>>(a, B); break;
    }
  } else {
    const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(uint64_t(N), kWarps), uint64_t(sms) * 8));
    switch (BT) {
      case 1: gemv_bf16_generic_kernel<1><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 2: gemv_bf16_generic_kernel<2><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 4: gemv_bf16_generic_kernel<4><<<blocks, kThreads, 0, s>>>(a, B); break;
      case 8: gemv_bf16_generic_kernel<8><<<blocks, kThreads, 0, s>>>(a, B); break;
      default: gemv_bf16_generic_kernel<16><<<blocks, kThreads, 0, s>>>(a, B); break;
    }
  }
  count_launches(1);
  return map_cuda(cudaGetLastError());
}
