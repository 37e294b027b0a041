// Encoder: histogram -> top-15 table -> pack codes and raw bits -> tile scan
// -> escape compaction -> row index.  All steps run on the GPU; the host reads
// back the escape count once to size the escape stream.
//
// Method: forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un
// 25%", section "Cómo funciona la compresión" (frequent sign+exponent symbols
// get 4-bit codes into a 15-entry table, rare symbols go to an exact escape
// stream, the low byte / 7-bit mantissa is stored unchanged).
#include <string.h>

#include <algorithm>

#include "wcomp_impl.cuh"

namespace wc {
namespace {

constexpr int kThreads = 256;  // pack / compact: one 8192-element tile per CTA

// ---------------------------------------------------------------------------
// a1: per-tensor histogram.  Each lane owns a column of a [bins][32] counter
// array in shared memory, so the 32 lanes of a warp never hit the same bank;
// different warps meet only through shared-memory atomics.
// ---------------------------------------------------------------------------
template <int SHIFT, int NB>
__global__ void __launch_bounds__(256) hist_kernel(const uint16_t* __restrict__ w, uint64_t n, int aligned,
                                                   uint32_t* __restrict__ hist) {
  extern __shared__ uint32_t h[];  // [NB][32]
  for (int i = threadIdx.x; i < NB * 32; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint64_t chunks = cdiv(n, 8);
  for (uint64_t ch = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; ch < chunks;
       ch += uint64_t(gridDim.x) * blockDim.x) {
    const uint64_t base = ch * 8;
    if (aligned && base + 8 <= n) {
      uint4 v = ld_stream_v4(w + base);
      uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        atomicAdd(&h[((wd[j] & 0xFFFF) >> SHIFT) * 32 + lane], 1u);
        atomicAdd(&h[(wd[j] >> (16 + SHIFT)) * 32 + lane], 1u);
      }
    } else {
      for (uint64_t i = base; i < n && i < base + 8; ++i) atomicAdd(&h[(uint32_t(w[i]) >> SHIFT) * 32 + lane], 1u);
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < NB; b += blockDim.x) {
    uint32_t s = 0;
    for (int l = 0; l < 32; ++l) s += h[b * 32 + ((l + b) & 31)];
    if (s) atomicAdd(&hist[b], s);
  }
}

// ---------------------------------------------------------------------------
// a2: table of the 15 most frequent symbols, ordered by (count desc, symbol
// asc), and the inverse map symbol -> code (15 = escape).  One CTA: every bin
// computes its rank by comparing against all bins.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512) select_kernel(const uint32_t* __restrict__ hist, int nb,
                                                     uint8_t* __restrict__ lut, uint16_t* __restrict__ table16) {
  __shared__ uint32_t cnt[kMaxBins];
  const int i = threadIdx.x;
  if (i < nb) cnt[i] = hist[i];
  if (i < 16) table16[i] = 0;
  __syncthreads();
  if (i < nb) {
    const uint32_t ci = cnt[i];
    int rank = 0;
    for (int j = 0; j < nb; ++j) {
      const uint32_t cj = cnt[j];
      rank += (cj > ci) || (cj == ci && j < i);
    }
    lut[i] = rank < kTableSize ? uint8_t(rank) : uint8_t(kEscape);
    if (rank < kTableSize) table16[rank] = uint16_t(i);
  }
}

__device__ __forceinline__ uint32_t block_sum_256(uint32_t v, uint32_t* sm) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t t = 0;
  if (threadIdx.x == 0)
    for (int k = 0; k < kThreads / 32; ++k) t += sm[k];
  return t;  // valid in thread 0
}

// Exclusive prefix of v over the 256 threads of the block (and the block total).
__device__ __forceinline__ uint32_t block_exclusive_256(uint32_t v, uint32_t* sm, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  uint32_t before = 0;
  total = 0;
  for (int k = 0; k < kThreads / 32; ++k) {
    const uint32_t s = sm[k];
    if (k < warp) before += s;
    total += s;
  }
  return before + inc - v;
}

// ---------------------------------------------------------------------------
// a3: pack.  Thread j of tile t handles group g = 256 t + j (32 elements).
// Writes the 16 code bytes, the raw bytes (byte-split) or the three mantissa
// planes (K15), and the tile's escape count.
// ---------------------------------------------------------------------------
template <int SCHEME>
__global__ void __launch_bounds__(kThreads) pack_kernel(const uint16_t* __restrict__ w, uint64_t n, int aligned,
                                                        const uint8_t* __restrict__ lut_g, uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ raw, uint8_t* __restrict__ pa,
                                                        uint8_t* __restrict__ pb, uint8_t* __restrict__ pc,
                                                        uint32_t* __restrict__ tile_counts) {
  __shared__ uint8_t lut[kMaxBins];
  __shared__ uint32_t red[kThreads / 32];
  constexpr int NB = SCHEME == WCOMP_BYTESPLIT ? 256 : 512;
  constexpr int SHIFT = SCHEME == WCOMP_BYTESPLIT ? 8 : 7;
  for (int i = threadIdx.x; i < NB; i += blockDim.x) lut[i] = lut_g[i];
  __syncthreads();
  const uint64_t G = cdiv(n, kGroup);
  const uint64_t g = uint64_t(blockIdx.x) * kThreads + threadIdx.x;
  uint32_t esc = 0;
  if (g < G) {
    const uint64_t base = g * kGroup;
    uint32_t wv[16];
    if (aligned && base + kGroup <= n) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 v = ld_stream_v4(w + base + 8 * k);
        wv[4 * k + 0] = v.x; wv[4 * k + 1] = v.y; wv[4 * k + 2] = v.z; wv[4 * k + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint64_t i0 = base + 2 * k;
        uint32_t lo = i0 < n ? w[i0] : 0u, hi = i0 + 1 < n ? w[i0 + 1] : 0u;
        wv[k] = lo | (hi << 16);
      }
    }
    uint32_t cw[4] = {0, 0, 0, 0};
    uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t a[4] = {0, 0, 0, 0}, b[2] = {0, 0}, c = 0;
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      const uint32_t v = (wv[e >> 1] >> (16 * (e & 1))) & 0xFFFF;
      const bool valid = base + e < n;
      uint32_t code = lut[v >> SHIFT];
      code = valid ? code : 0u;
      esc += (code == kEscape);
      cw[e >> 3] |= code << (4 * (e & 7));
      const int q = e >> 2, ln = e & 3;
      if (SCHEME == WCOMP_BYTESPLIT) {
        r[e >> 2] |= (valid ? (v & 0xFF) : 0u) << (8 * (e & 3));
      } else {
        const uint32_t m = valid ? (v & 0x7F) : 0u;
        a[q >> 1] |= (m & 0xF) << (8 * ln + 4 * (q & 1));
        b[q >> 2] |= ((m >> 4) & 0x3) << (8 * ln + 2 * (q & 3));
        c |= ((m >> 6) & 0x1) << (8 * ln + q);
      }
    }
    *reinterpret_cast<uint4*>(codes + 16 * g) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    if (SCHEME == WCOMP_BYTESPLIT) {
      *reinterpret_cast<uint4*>(raw + 32 * g) = make_uint4(r[0], r[1], r[2], r[3]);
      if (base + 16 < n) *reinterpret_cast<uint4*>(raw + 32 * g + 16) = make_uint4(r[4], r[5], r[6], r[7]);
    } else {
      *reinterpret_cast<uint4*>(pa + 16 * g) = make_uint4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<uint2*>(pb + 8 * g) = make_uint2(b[0], b[1]);
      *reinterpret_cast<uint32_t*>(pc + 4 * g) = c;
    }
  }
  const uint32_t total = block_sum_256(esc, red);
  if (threadIdx.x == 0) tile_counts[blockIdx.x] = total;
}

// ---------------------------------------------------------------------------
// Exclusive scan of the per-tile escape counts, in place; entry n_tiles
// receives E.  One CTA, two passes, no inter-block waits.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) scan_kernel(uint32_t* __restrict__ idx, uint32_t n_tiles) {
  __shared__ uint32_t part[1024];
  const uint32_t per = uint32_t(cdiv(n_tiles, 1024));
  const uint32_t lo = threadIdx.x * per;
  const uint32_t hi = min(lo + per, n_tiles);
  uint32_t s = 0;
  for (uint32_t i = lo; i < hi; ++i) s += idx[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    uint32_t v = threadIdx.x >= unsigned(o) ? part[threadIdx.x - o] : 0u;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  uint32_t run = part[threadIdx.x] - s;
  for (uint32_t i = lo; i < hi; ++i) {
    const uint32_t v = idx[i];
    idx[i] = run;
    run += v;
  }
  if (threadIdx.x == 1023) idx[n_tiles] = part[1023];
}

// ---------------------------------------------------------------------------
// a4: escape compaction.  Thread j of tile t re-reads the 32 codes of group
// 256 t + j, ranks its escapes inside the tile with a block scan and writes
// (position, value) pairs in ascending position order.
// ---------------------------------------------------------------------------
template <int SCHEME>
__global__ void __launch_bounds__(kThreads) compact_kernel(const uint16_t* __restrict__ w, uint64_t n,
                                                           const uint8_t* __restrict__ codes,
                                                           const uint32_t* __restrict__ tile_index,
                                                           uint32_t* __restrict__ pos, uint8_t* __restrict__ val) {
  __shared__ uint32_t sm[kThreads / 32];
  const uint32_t t = blockIdx.x;
  if (tile_index[t + 1] == tile_index[t]) return;  // uniform: no escapes in this tile
  const uint64_t G = cdiv(n, kGroup);
  const uint64_t g = uint64_t(t) * kThreads + threadIdx.x;
  uint4 c4 = make_uint4(0, 0, 0, 0);
  if (g < G) c4 = *reinterpret_cast<const uint4*>(codes + 16 * g);
  const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
  uint32_t cnt = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = cw[i] & (cw[i] >> 1) & (cw[i] >> 2) & (cw[i] >> 3) & 0x11111111u;
    cnt += __popc(x);
  }
  uint32_t total;
  uint32_t o = tile_index[t] + block_exclusive_256(cnt, sm, total);
  if (!cnt) return;
  const uint64_t base = g * kGroup;
  for (int e = 0; e < kGroup; ++e) {
    if (((cw[e >> 3] >> (4 * (e & 7))) & 0xF) == kEscape) {
      const uint32_t p = uint32_t(base + e);
      const uint32_t v = w[p];
      pos[o] = p;
      if (SCHEME == WCOMP_BYTESPLIT)
        val[o] = uint8_t(v >> 8);
      else
        reinterpret_cast<uint16_t*>(val)[o] = uint16_t(v);
      ++o;
    }
  }
}

// Row index: entry r = number of escapes below r * K (lower bound search).
__global__ void row_index_kernel(const uint32_t* __restrict__ pos, uint64_t E, int64_t N, int64_t K,
                                 uint32_t* __restrict__ row_index) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r > N) return;
  const uint64_t bound = uint64_t(r) * uint64_t(K);
  uint64_t lo = 0, hi = E;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) >> 1;
    if (pos[mid] < bound) lo = mid + 1; else hi = mid;
  }
  row_index[r] = uint32_t(lo);
}

cudaError_t zero_pad(uint8_t* base, uint64_t off, uint64_t sz, cudaStream_t s) {
  const uint64_t p = padsec(sz);
  if (p == sz) return cudaSuccess;
  return cudaMemsetAsync(base + off + sz, 0, p - sz, s);
}

}  // namespace
}  // namespace wc

using namespace wc;

extern "C" int wcomp_encode(const uint16_t* d_w, int64_t N, int64_t K, int scheme, void* stream,
                            wcomp_container** out) {
  if (!out) return WCOMP_EINVAL;
  *out = nullptr;
  if (!d_w || N <= 0 || K <= 0) return WCOMP_EINVAL;
  if (scheme != WCOMP_BYTESPLIT && scheme != WCOMP_K15) return WCOMP_EINVAL;
  if (N >= (int64_t(1) << 32) || K >= (int64_t(1) << 32) || uint64_t(N) * uint64_t(K) >= (uint64_t(1) << 32))
    return WCOMP_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wcomp_container* c = new (std::nothrow) wcomp_container();
  if (!c) return WCOMP_ENOMEM;
  cudaGetDevice(&c->device);
  Layout& L = c->L;
  L.compute(scheme, N, K, 0);
  const int aligned = (reinterpret_cast<uintptr_t>(d_w) & 15) == 0;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&c->d_main), L.main_alloc, s);
  if (e != cudaSuccess) {
    delete c;
    return map_cuda(e);
  }
  uint8_t* m = c->d_main;
  uint32_t* hist = reinterpret_cast<uint32_t*>(m + L.off_scratch + Scratch::hist);
  uint8_t* lut = m + L.off_scratch + Scratch::lut;
  uint16_t* table16 = reinterpret_cast<uint16_t*>(m + L.off_scratch + Scratch::table);
  uint32_t* tile_idx = reinterpret_cast<uint32_t*>(m + L.off_tile);
  uint32_t* row_idx = reinterpret_cast<uint32_t*>(m + L.off_row);
  const int nb = scheme == WCOMP_BYTESPLIT ? 256 : 512;

  e = cudaMemsetAsync(hist, 0, kMaxBins * sizeof(uint32_t), s);
  if (e == cudaSuccess) e = zero_pad(m, L.off_b, L.sz_b, s);
  if (e == cudaSuccess) e = zero_pad(m, L.off_c, L.sz_c, s);
  if (e == cudaSuccess) e = zero_pad(m, L.off_tile, L.sz_tile, s);
  if (e == cudaSuccess) e = zero_pad(m, L.off_row, L.sz_row, s);

  const int sms = sm_count(c->device);
  if (e == cudaSuccess) {
    const uint64_t chunks = cdiv(L.n, 8);
    const int grid = int(std::min<uint64_t>(cdiv(chunks, 256), uint64_t(sms) * 4));
    if (scheme == WCOMP_BYTESPLIT) {
      const size_t smem = 256 * 32 * sizeof(uint32_t);
      hist_kernel<8, 256><<<grid, 256, smem, s>>>(d_w, L.n, aligned, hist);
    } else {
      const size_t smem = 512 * 32 * sizeof(uint32_t);
      static bool attr = false;
      if (!attr) {
        cudaFuncSetAttribute(hist_kernel<7, 512>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        attr = true;
      }
      hist_kernel<7, 512><<<grid, 256, smem, s>>>(d_w, L.n, aligned, hist);
    }
    select_kernel<<<1, 512, 0, s>>>(hist, nb, lut, table16);
    const unsigned tiles = unsigned(L.n_tiles);
    if (scheme == WCOMP_BYTESPLIT)
      pack_kernel<WCOMP_BYTESPLIT><<<tiles, kThreads, 0, s>>>(d_w, L.n, aligned, lut, m + L.off_codes,
                                                              m + L.off_raw, nullptr, nullptr, nullptr, tile_idx);
    else
      pack_kernel<WCOMP_K15><<<tiles, kThreads, 0, s>>>(d_w, L.n, aligned, lut, m + L.off_codes, nullptr,
                                                        m + L.off_a, m + L.off_b, m + L.off_c, tile_idx);
    scan_kernel<<<1, 1024, 0, s>>>(tile_idx, tiles);
    count_launches(4);  // histogram, select, pack, scan
    e = cudaGetLastError();
  }
  struct {
    uint32_t E;
    uint16_t table[16];
  } hostinfo;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hostinfo.E, tile_idx + L.n_tiles, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(hostinfo.table, table16, 32, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    wcomp_free(c, stream);
    return map_cuda(e);
  }
  memcpy(c->table, hostinfo.table, sizeof(c->table));
  L.compute(scheme, N, K, hostinfo.E);
  if (L.E) {
    e = cudaMallocAsync(reinterpret_cast<void**>(&c->d_esc), L.esc_payload, s);
    uint8_t* x = c->d_esc;
    if (e == cudaSuccess) e = zero_pad(x, L.off_pos, L.sz_pos, s);
    if (e == cudaSuccess) e = zero_pad(x, L.off_val, L.sz_val, s);
    if (e == cudaSuccess) {
      uint32_t* pos = reinterpret_cast<uint32_t*>(x + L.off_pos);
      uint8_t* val = x + L.off_val;
      if (scheme == WCOMP_BYTESPLIT)
        compact_kernel<WCOMP_BYTESPLIT><<<unsigned(L.n_tiles), kThreads, 0, s>>>(d_w, L.n, m + L.off_codes,
                                                                                tile_idx, pos, val);
      else
        compact_kernel<WCOMP_K15><<<unsigned(L.n_tiles), kThreads, 0, s>>>(d_w, L.n, m + L.off_codes, tile_idx,
                                                                          pos, val);
      row_index_kernel<<<unsigned(cdiv(uint64_t(N) + 1, 256)), 256, 0, s>>>(pos, L.E, N, K, row_idx);
      count_launches(2);  // compact, row index
      e = cudaGetLastError();
    }
  } else {
    e = cudaMemsetAsync(row_idx, 0, 4 * (uint64_t(N) + 1), s);
  }
  if (e != cudaSuccess) {
    wcomp_free(c, stream);
    return map_cuda(e);
  }
  *out = c;
  return WCOMP_OK;
}
