// Standalone decode: container -> exact BF16 in HBM, for one tensor or a batch
// of tensors in a single launch.
//
// Method: forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un
// 25%", section "Cómo funciona la compresión" (byte-split rebuilds the high
// byte from the dictionary codes and the escape stream and keeps the low byte;
// K15 rebuilds the 9-bit symbol and appends the raw 7-bit mantissa).
//
// One CTA of 256 threads decodes one 8192-element tile: thread j expands the
// 32 codes of its group through the register table (prmt lookups), joins the
// raw bytes / mantissa planes, and writes 64 bytes with two 256-bit stores.
// Escaped elements first receive the placeholder symbol 0; after a CTA
// barrier the threads write the tile's escapes over them, one entry each,
// from the tile's slice of the escape stream (found in O(1) through the tile
// index).
#include <string.h>

#include <algorithm>

#include "wcomp_impl.cuh"

namespace wc {
namespace {
WCOMP_DEBUG_WORD

constexpr int kThreads = 256;

template <int SCHEME>
__device__ __forceinline__ void decode_tile(const TensorDesc& d, uint16_t* __restrict__ out, uint32_t tile) {
  const uint64_t G = cdiv(d.n, kGroup);
  const uint64_t g = uint64_t(tile) * kThreads + threadIdx.x;
  if (g < G) {
    const uint64_t base = g * kGroup;
    if (d.aligned && base + kGroup <= d.n) {
      uint32_t cw[4], r[8], o[16];
      load_group<SCHEME>(d, g, cw, r);
      decode_group<SCHEME>(d.t, cw, r, o);
      st_v8(out + base, o);
      st_v8(out + base + 16, o + 8);
    } else {
      for (uint64_t i = base; i < d.n && i < base + kGroup; ++i) out[i] = uint16_t(decode_elem_placeholder(d, i));
    }
  }
  const uint32_t e0 = d.tile_index[tile], e1 = d.tile_index[tile + 1];
  if (e0 == e1) return;  // the same for every thread of the CTA
  // The CTA's threads share the tile's escape slice, one entry each: a CTA
  // barrier orders every placeholder store of the tile before the patches.
  __syncthreads();
  for (uint32_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
    if (!WCOMP_DCHECK(e < d.E, 0)) continue;
    const uint32_t p = d.esc_pos[e];
    if (!WCOMP_DCHECK(p < d.n && p / kTile == tile, 0)) continue;
    out[p] = d.esc_val[e];  // the whole word
  }
}

__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeBatch p,
                                                          uint32_t total_tiles) {
  for (uint32_t gt = blockIdx.x; gt < total_tiles; gt += gridDim.x) {
    int i = 0;
    while (i + 1 < p.count && p.tile_prefix[i + 1] <= gt) ++i;
    const TensorDesc& d = p.d[i];
    const uint32_t tile = gt - p.tile_prefix[i];
    if (d.scheme == WCOMP_BYTESPLIT)
      decode_tile<WCOMP_BYTESPLIT>(d, p.out[i], tile);
    else
      decode_tile<WCOMP_K15>(d, p.out[i], tile);
  }
}

int launch_decode(const wcomp_container* const* cs, uint16_t* const* outs, int count, cudaStream_t s) {
  for (int i = 0; i < count; ++i)
    if (!cs[i] || !outs[i]) return WCOMP_EINVAL;
  for (int start = 0; start < count; start += kMaxBatch) {
    const int m = std::min(kMaxBatch, count - start);
    DecodeBatch b;
    memset(&b, 0, sizeof(b));
    b.count = m;
    uint64_t tiles = 0;
    for (int j = 0; j < m; ++j) {
      const wcomp_container* c = cs[start + j];
      b.d[j] = make_desc(c);
      b.d[j].aligned = ((reinterpret_cast<uintptr_t>(outs[start + j]) | reinterpret_cast<uintptr_t>(c->d_main)) & 31) == 0;
      b.out[j] = outs[start + j];
      b.tile_prefix[j] = uint32_t(tiles);
      tiles += c->L.n_tiles;
      if (tiles >= (uint64_t(1) << 31)) return WCOMP_EUNSUPPORTED;
    }
    b.tile_prefix[m] = uint32_t(tiles);
    // one CTA per tile: the hardware hands each finished CTA's slot to the next
    // tile, so no SM idles behind a CTA's last tile (a grid of eight CTAs per SM
    // looping over tiles took one layer's decode, both schemes, from 0.575 to
    // 0.633 ms)
    const uint32_t grid = uint32_t(tiles);
    decode_kernel<<<grid, kThreads, 0, s>>>(b, uint32_t(tiles));
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return map_cuda(e);
  }
  return WCOMP_OK;
}

}  // namespace

WCOMP_DEBUG_TAKE(debug_take_decode)
}  // namespace wc

using namespace wc;

extern "C" int wcomp_decode(const wcomp_container* c, uint16_t* d_out, void* stream) {
  if (!c || !d_out) return WCOMP_EINVAL;
  return launch_decode(&c, &d_out, 1, static_cast<cudaStream_t>(stream));
}

extern "C" int wcomp_decode_batched(const wcomp_container* const* containers, uint16_t* const* d_outs, int count,
                                    void* stream) {
  if (!containers || !d_outs || count <= 0) return WCOMP_EINVAL;
  return launch_decode(containers, d_outs, count, static_cast<cudaStream_t>(stream));
}
