// Encoder: histogram -> top-15 table -> pack codes and raw bits -> tile scan
// -> escape compaction -> row index, for one tensor or a batch of tensors.
// All steps run on the GPU; the host reads back the tables and escape counts
// once per batch (right after the table selection) to size the escape streams.
//
// Method: forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un
// 25%", section "Cómo funciona la compresión" (frequent sign+exponent symbols
// get 4-bit codes into a 15-entry table, rare symbols go to an exact escape
// stream, the low byte / 7-bit mantissa is stored unchanged).
//
// Every kernel takes the whole batch as a parameter-space descriptor array
// and finds its tensor from a prefix over blocks, tiles or rows, so a batch
// costs about a dozen launches and one host synchronization.  The pack pass
// stashes each tile's escapes while it holds the source words, so the
// compaction pass only moves E entries instead of reading the source again.
#include <string.h>

#include <algorithm>
#include <vector>

#include "wcomp_impl.cuh"

namespace wc {
namespace {
WCOMP_DEBUG_WORD

constexpr int kThreads = 256;  // pack / compact: one 8192-element tile per CTA

struct Summary {
  uint32_t E;         // escapes implied by the histogram: n minus the table symbols' counts
  uint16_t table[16];
  uint32_t scanned;   // escapes the pack pass actually found (the tile scan's total)
  uint32_t pad[2];
};

struct EncDesc {
  const uint16_t* w;
  uint8_t* main;
  uint8_t* esc;
  Summary* summary;
  const uint32_t* hist_k15;  // byte-split job whose K15 twin is in the batch: fold that histogram
  uint32_t* stash_pos;  // per tile: up to stash_cap escapes found by pack, in tile order
  uint16_t* stash_val;
  uint32_t stash_cap;
  uint64_t n;
  int64_t N, K;
  uint64_t E;
  uint64_t off_codes, off_raw, off_a, off_b, off_c, off_tile, off_row, off_scratch, off_pos, off_val;
  uint32_t n_tiles;
  int scheme;
  int aligned;
};

struct EncBatch {
  EncDesc d[kMaxBatch];
  uint32_t prefix[kMaxBatch + 1];  // blocks, tiles or rows, per launch
  int count;
};

constexpr int kMaxZero = 8 * kMaxBatch;
struct ZeroList {
  uint8_t* p[kMaxZero];
  uint32_t len[kMaxZero];
  int count;
};

// The last of entries 0 .. count - 1 whose prefix is at most x (binary search).
__device__ __forceinline__ int owner_in(const uint32_t* prefix, int count, uint32_t x) {
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int find_owner(const EncBatch& b, uint32_t x) { return owner_in(b.prefix, b.count, x); }

// Zero small byte ranges (section padding, histogram scratch); one CTA per range.
__global__ void __launch_bounds__(256) zero_kernel(const __grid_constant__ ZeroList z) {
  const int r = blockIdx.x;
  if (r >= z.count) return;
  uint8_t* p = z.p[r];
  for (uint32_t i = threadIdx.x; i < z.len[r]; i += blockDim.x) p[i] = 0;
}

// ---------------------------------------------------------------------------
// a1: per-tensor histogram.  Counters live in shared memory as [bins][16]
// words; lane l owns the low half of column l (l < 16) or the high half of
// column l - 16, so the lanes of a warp touch 16 distinct banks and two lanes
// share a word only as its two halves.  A half therefore collects the counts
// of 8 threads (one lane of each warp).  Work is dealt out in 8-element
// chunks, so a thread meets at most 8 x (its chunk count) elements; the host
// (hist_blocks) sizes the grid so that no thread gets more than
// kHistMaxChunks chunks: 8 threads x 8 x 1023 = 65472 < 65536, so a half
// cannot wrap even when every element has the same symbol.
// ---------------------------------------------------------------------------
constexpr uint64_t kHistMaxChunks = 1023;
constexpr uint32_t kHistThreads = 256;
template <int SHIFT, int NB>
__global__ void __launch_bounds__(256) hist_kernel(const __grid_constant__ EncBatch bt) {
  __shared__ uint32_t h[NB * 16];
  for (int i = threadIdx.x; i < NB * 16; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int t = find_owner(bt, blockIdx.x);
  const EncDesc& d = bt.d[t];
  const uint32_t blk = blockIdx.x - bt.prefix[t], nblk = bt.prefix[t + 1] - bt.prefix[t];
  const int lane = threadIdx.x & 31;
  const uint32_t col = lane & 15, inc = lane < 16 ? 1u : 65536u;
  const uint64_t chunks = cdiv(d.n, 8);
  const uint64_t stride = uint64_t(nblk) * blockDim.x;
  const uint64_t full = d.aligned ? d.n / 8 : 0;  // chunks of 8 that take one 16-byte load
  uint64_t ch = uint64_t(blk) * blockDim.x + threadIdx.x;
  // four loads in flight before their counts
  for (; ch + 3 * stride < full; ch += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ld_stream_v4(d.w + (ch + u * stride) * 8);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        atomicAdd(&h[((wd[j] & 0xFFFF) >> SHIFT) * 16 + col], inc);
        atomicAdd(&h[(wd[j] >> (16 + SHIFT)) * 16 + col], inc);
      }
    }
  }
  for (; ch < chunks; ch += stride) {
    const uint64_t base = ch * 8;
    if (ch < full) {
      const uint4 v = ld_stream_v4(d.w + base);
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        atomicAdd(&h[((wd[j] & 0xFFFF) >> SHIFT) * 16 + col], inc);
        atomicAdd(&h[(wd[j] >> (16 + SHIFT)) * 16 + col], inc);
      }
    } else {
      for (uint64_t i = base; i < d.n && i < base + 8; ++i)
        atomicAdd(&h[(uint32_t(d.w[i]) >> SHIFT) * 16 + col], inc);
    }
  }
  __syncthreads();
  uint32_t* hist = reinterpret_cast<uint32_t*>(d.main + d.off_scratch + Scratch::hist);
  for (int b = threadIdx.x; b < NB; b += blockDim.x) {
    uint32_t s = 0;
    for (int l = 0; l < 16; ++l) {
      const uint32_t v = h[b * 16 + ((l + b) & 15)];
      s += (v & 0xFFFF) + (v >> 16);
    }
    if (s) atomicAdd(&hist[b], s);
  }
}

// ---------------------------------------------------------------------------
// a2: table of the 15 most frequent symbols, ordered by (count desc, symbol
// asc), and the inverse map symbol -> code (15 = escape).  One CTA per tensor:
// every bin computes its rank by comparing against all bins.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512) select_kernel(const __grid_constant__ EncBatch bt) {
  __shared__ uint32_t cnt[kMaxBins];
  __shared__ unsigned long long coded;
  const EncDesc& d = bt.d[blockIdx.x];
  const int nb = d.scheme == WCOMP_BYTESPLIT ? 256 : 512;
  const uint32_t* hist = reinterpret_cast<const uint32_t*>(d.main + d.off_scratch + Scratch::hist);
  uint8_t* lut = d.main + d.off_scratch + Scratch::lut;
  const int i = threadIdx.x;
  if (i < nb) {
    // a byte-split symbol is a K15 symbol without its exponent LSB: bins 2s and 2s+1 fold into s
    cnt[i] = d.hist_k15 ? d.hist_k15[2 * i] + d.hist_k15[2 * i + 1] : hist[i];
  }
  if (i < 16) d.summary->table[i] = 0;
  if (i == 0) coded = 0;
  __syncthreads();
  if (i < nb) {
    const uint32_t ci = cnt[i];
    int rank = 0;
    for (int j = 0; j < nb; ++j) {
      const uint32_t cj = cnt[j];
      rank += (cj > ci) || (cj == ci && j < i);
    }
    lut[i] = rank < kTableSize ? uint8_t(rank) : uint8_t(kEscape);
    if (rank < kTableSize) {
      d.summary->table[rank] = uint16_t(i);
      atomicAdd(&coded, (unsigned long long)ci);
    }
  }
  __syncthreads();
  if (i == 0) d.summary->E = uint32_t(d.n - coded);  // every symbol outside the table escapes
}

// Exclusive prefix of v over the 256 threads of the block (sm: 8 words).
__device__ __forceinline__ uint32_t block_exclusive_256(uint32_t v, uint32_t* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  uint32_t before = 0;
  for (int k = 0; k < warp; ++k) before += sm[k];
  return before + inc - v;
}

__device__ __forceinline__ uint32_t block_total_256(const uint32_t* sm) {
  uint32_t t = 0;
  for (int k = 0; k < kThreads / 32; ++k) t += sm[k];
  return t;
}

// ---------------------------------------------------------------------------
// a3: pack.  Thread j of a tile handles group 256 t + j (32 elements): the 16
// code bytes, the raw bytes (byte-split) or the three mantissa planes (K15),
// and the tile's escape count.
// ---------------------------------------------------------------------------

// The group's 32 source elements as 16 element-pair words (zero past n).
__device__ __forceinline__ void load_group(const EncDesc& d, uint64_t g, uint32_t (&wv)[16]) {
  const uint64_t n = d.n, base = g * kGroup;
  if (d.aligned && base + kGroup <= n) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = ld_stream_v4(d.w + base + 8 * k);
      wv[4 * k + 0] = v.x; wv[4 * k + 1] = v.y; wv[4 * k + 2] = v.z; wv[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint64_t i0 = base + 2 * k;
      const uint32_t lo = i0 < n ? d.w[i0] : 0u, hi = i0 + 1 < n ? d.w[i0 + 1] : 0u;
      wv[k] = lo | (hi << 16);
    }
  }
}

template <int SCHEME>
__device__ __forceinline__ void load_lut(const EncDesc& d, uint8_t* lut) {
  constexpr int NB = SCHEME == WCOMP_BYTESPLIT ? 256 : 512;
  const uint8_t* lut_g = d.main + d.off_scratch + Scratch::lut;
  for (int i = threadIdx.x; i < NB; i += blockDim.x) lut[i] = lut_g[i];
}

// Codes (cw: element e at bits 4 (e mod 8) of cw[e / 8]) and raw bytes /
// planes of group g, written to the container; returns the escape count.
template <int SCHEME>
__device__ __forceinline__ void group_codes(const uint8_t* lut, const uint32_t (&wv)[16], uint32_t (&cw)[4]) {
  constexpr int NB = SCHEME == WCOMP_BYTESPLIT ? 256 : 512;
  constexpr int SHIFT = SCHEME == WCOMP_BYTESPLIT ? 8 : 7;
  cw[0] = cw[1] = cw[2] = cw[3] = 0u;
  // the symbol of an element pair word is bits 8.. (byte-split) or 7.. (K15) of each half
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t s0 = (wv[k] >> SHIFT) & (NB - 1), s1 = wv[k] >> (16 + SHIFT);
    const uint32_t c0 = lut[s0], c1 = lut[s1];
    cw[k >> 2] += (c0 | (c1 << 4)) << (8 * (k & 3));
  }
}

// Bit 4j + 3 set where nibble j of c is 15: its low three bits plus one carry
// into bit 3, which must also be set.
__device__ __forceinline__ uint32_t nibbles15(uint32_t c) {
  return ((c & 0x77777777u) + 0x11111111u) & c & 0x88888888u;
}

// Codes in cw are given; clears codes past n, writes the group's sections
// and returns its escape count.
template <int SCHEME>
__device__ __forceinline__ uint32_t pack_group(const EncDesc& d, uint64_t g, const uint32_t (&lo)[8],
                                               uint32_t (&cw)[4]) {
  const uint64_t n = d.n, base = g * kGroup;
  if (base + kGroup > n) {
    // the tensor's last group: elements past n get code 0 (the source words were zero-filled)
    const uint32_t valid = uint32_t(n - base);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int keep = int(valid) - 8 * k;
      cw[k] &= keep >= 8 ? 0xFFFFFFFFu : keep <= 0 ? 0u : (1u << (4 * keep)) - 1u;
    }
  }
  uint32_t esc = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) esc += __popc(nibbles15(cw[k]));
  uint8_t* m = d.main;
  *reinterpret_cast<uint4*>(m + d.off_codes + 16 * g) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  if (SCHEME == WCOMP_BYTESPLIT) {
    *reinterpret_cast<uint4*>(m + d.off_raw + 32 * g) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (base + 16 < n) *reinterpret_cast<uint4*>(m + d.off_raw + 32 * g + 16) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  } else {
    // K15 mantissa bytes from the low bytes (bit 7 of a low byte is the
    // exponent bit and is dropped): word q < 7 is quad q's four mantissas
    // with bit 7 of byte lane i carrying bit q of element 28 + i's mantissa
    uint32_t a[4], b[2], c;
    uint32_t wq[7];
#pragma unroll
    for (int q = 0; q < 7; ++q) wq[q] = (lo[q] & 0x7F7F7F7Fu) | (((lo[7] >> q) << 7) & 0x80808080u);
    a[0] = wq[0]; a[1] = wq[1]; a[2] = wq[2]; a[3] = wq[3];
    b[0] = wq[4]; b[1] = wq[5];
    c = wq[6];
    *reinterpret_cast<uint4*>(m + d.off_a + 16 * g) = make_uint4(a[0], a[1], a[2], a[3]);
    *reinterpret_cast<uint2*>(m + d.off_b + 8 * g) = make_uint2(b[0], b[1]);
    *reinterpret_cast<uint32_t*>(m + d.off_c + 4 * g) = c;
  }
  return esc;
}

// Stash (position, value) of the group's escapes at slots before.. of the
// tile's stash; visits only the set bits of each word's code-15 mask (codes
// past n were cleared, so every visited element is valid).
template <int SCHEME>
__device__ __forceinline__ void stash_group(const EncDesc& d, uint32_t tile, uint64_t g, uint32_t before,
                                            const uint32_t (&wv)[16], const uint32_t (&cw)[4]) {
  uint64_t o = uint64_t(tile) * d.stash_cap + before;
  const uint64_t base = g * kGroup;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t m = nibbles15(cw[k]);
    while (m) {
      const int j = (__ffs(m) - 1) >> 2;
      m &= m - 1;
      const uint32_t pw = (j >> 1) == 0 ? wv[4 * k] : (j >> 1) == 1 ? wv[4 * k + 1]
                          : (j >> 1) == 2 ? wv[4 * k + 2] : wv[4 * k + 3];
      const uint32_t v = (pw >> (16 * (j & 1))) & 0xFFFF;
      if (!WCOMP_DCHECK(o < uint64_t(tile + 1) * d.stash_cap && o < uint64_t(d.n_tiles) * d.stash_cap, 3)) break;
      d.stash_pos[o] = uint32_t(base + 8 * k + j);
      d.stash_val[o] = uint16_t(v);  // the whole word (the device keeps whole escape words)
      ++o;
    }
  }
}

template <int SCHEME>
__global__ void __launch_bounds__(kThreads) pack_kernel(const __grid_constant__ EncBatch bt) {
  __shared__ uint8_t lut[kMaxBins];
  __shared__ uint32_t red[kThreads / 32];
  const int ti = find_owner(bt, blockIdx.x);
  const EncDesc& d = bt.d[ti];
  const uint32_t tile = blockIdx.x - bt.prefix[ti];
  const uint64_t g = uint64_t(tile) * kThreads + threadIdx.x;
  const bool live = g < cdiv(d.n, kGroup);
  uint32_t wv[16], cw[4] = {0u, 0u, 0u, 0u}, esc = 0;
  // the source words are requested first, so their latency overlaps the
  // table's trip through shared memory
  if (live) load_group(d, g, wv);
  load_lut<SCHEME>(d, lut);
  __syncthreads();
  if (live) {
    uint32_t lo[8];  // low bytes of elements 4q .. 4q+3
#pragma unroll
    for (int q = 0; q < 8; ++q) lo[q] = prmt(wv[2 * q], wv[2 * q + 1], 0x6420);
    group_codes<SCHEME>(lut, wv, cw);
    esc = pack_group<SCHEME>(d, g, lo, cw);
  }
  // rank the escapes inside the tile; while the source words are still in
  // registers, stash (position, value) for the gather pass
  const uint32_t before = block_exclusive_256(esc, red);
  const uint32_t total = block_total_256(red);
  if (threadIdx.x == 0) reinterpret_cast<uint32_t*>(d.main + d.off_tile)[tile] = total;
  if (esc && total <= d.stash_cap) stash_group<SCHEME>(d, tile, g, before, wv, cw);
}

// Both schemes of one tensor in one pass: a tile is read once and packed
// into its byte-split and its K15 container.  bt.d[2i] is the byte-split job
// and bt.d[2i + 1] its K15 twin; bt.prefix counts tiles per pair.  The two
// escape counts share one block scan as 16-bit halves (a tile holds at most
// 8192 escapes per scheme).
// Five CTAs per SM (at most 48 registers): measured 2 % faster than the four
// that 58 registers allow, for one layer of the checkpoint-shaped set.
__global__ void __launch_bounds__(kThreads, 5) pack_twin_kernel(const __grid_constant__ EncBatch bt) {
  // one table for both: entry s (a K15 symbol) holds the K15 code of s in its
  // low nibble and the byte-split code of s >> 1 (the high byte) in its high
  // nibble, so one lookup per element gives both codes
  __shared__ uint8_t lut2[512];
  __shared__ uint32_t red[kThreads / 32];
  const int pi = owner_in(bt.prefix, bt.count / 2, blockIdx.x);
  const EncDesc& d0 = bt.d[2 * pi];
  const EncDesc& d1 = bt.d[2 * pi + 1];
  const uint32_t tile = blockIdx.x - bt.prefix[pi];
  const uint64_t g = uint64_t(tile) * kThreads + threadIdx.x;
  const bool live = g < cdiv(d0.n, kGroup);
  uint32_t wv[16], cw0[4] = {0u, 0u, 0u, 0u}, cw1[4] = {0u, 0u, 0u, 0u}, esc = 0;
  if (live) load_group(d1, g, wv);
  {
    const uint8_t* l0 = d0.main + d0.off_scratch + Scratch::lut;
    const uint8_t* l1 = d1.main + d1.off_scratch + Scratch::lut;
    for (int i = threadIdx.x; i < 512; i += blockDim.x) lut2[i] = uint8_t(l1[i] | (l0[i >> 1] << 4));
  }
  __syncthreads();
  if (live) {
    uint32_t lo[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) lo[q] = prmt(wv[2 * q], wv[2 * q + 1], 0x6420);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // table bytes of elements 8i .. 8i + 7, four to a word (byte lane = element)
      uint32_t T[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = wv[4 * i + 2 * h], w1 = wv[4 * i + 2 * h + 1];
        const uint32_t b0 = lut2[(w0 >> 7) & 511u], b1 = lut2[w0 >> 23];
        const uint32_t b2 = lut2[(w1 >> 7) & 511u], b3 = lut2[w1 >> 23];
        T[h] = prmt(prmt(b0, b1, 0x0040u), prmt(b2, b3, 0x0040u), 0x5410u);
      }
      // code word: byte j = element 2j | element 2j + 1 << 4.  K15 codes are
      // the low nibbles of the table bytes, byte-split codes the high nibbles.
      const uint32_t k0 = T[0] & 0x0F0F0F0Fu, k1 = T[1] & 0x0F0F0F0Fu;
      const uint32_t s0 = (T[0] >> 4) & 0x0F0F0F0Fu, s1 = (T[1] >> 4) & 0x0F0F0F0Fu;
      cw1[i] = prmt(k0 | (k0 >> 4), k1 | (k1 >> 4), 0x6420u);
      cw0[i] = prmt(s0 | (s0 >> 4), s1 | (s1 >> 4), 0x6420u);
    }
    esc = pack_group<WCOMP_BYTESPLIT>(d0, g, lo, cw0);
    esc |= pack_group<WCOMP_K15>(d1, g, lo, cw1) << 16;
  }
  const uint32_t before = block_exclusive_256(esc, red);
  const uint32_t total = block_total_256(red);
  if (threadIdx.x == 0) {
    reinterpret_cast<uint32_t*>(d0.main + d0.off_tile)[tile] = total & 0xFFFF;
    reinterpret_cast<uint32_t*>(d1.main + d1.off_tile)[tile] = total >> 16;
  }
  if ((esc & 0xFFFF) && (total & 0xFFFF) <= d0.stash_cap)
    stash_group<WCOMP_BYTESPLIT>(d0, tile, g, before & 0xFFFF, wv, cw0);
  if ((esc >> 16) && (total >> 16) <= d1.stash_cap) stash_group<WCOMP_K15>(d1, tile, g, before >> 16, wv, cw1);
}

// ---------------------------------------------------------------------------
// Exclusive scan of the per-tile escape counts, in place; entry n_tiles
// receives E.  One CTA per tensor, two passes, no inter-block waits.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) scan_kernel(const __grid_constant__ EncBatch bt) {
  __shared__ uint32_t part[1024];
  const EncDesc& d = bt.d[blockIdx.x];
  uint32_t* idx = reinterpret_cast<uint32_t*>(d.main + d.off_tile);
  const uint32_t n_tiles = d.n_tiles;
  const uint32_t per = uint32_t(cdiv(n_tiles, 1024));
  const uint32_t lo = threadIdx.x * per;
  const uint32_t hi = min(lo + per, n_tiles);
  uint32_t s = 0;
  for (uint32_t i = lo; i < hi; ++i) s += idx[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const uint32_t v = threadIdx.x >= unsigned(o) ? part[threadIdx.x - o] : 0u;
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
  if (threadIdx.x == 1023) {
    idx[n_tiles] = part[1023];
    d.summary->scanned = part[1023];  // checked on the host against the histogram's E
  }
}

// ---------------------------------------------------------------------------
// a4: escape compaction.  A tile whose escapes fit its stash copies them to
// their final place (tile_index[t] onwards).  A tile with more escapes than
// the stash holds is ranked again here: thread j re-reads the 32 codes of its
// group, a block scan gives each escape its place, and the values are read
// back from the source.  Either way the stream ends up in ascending position
// order.
//
// A CTA covers kCompactTiles consecutive tiles of one tensor: warp w copies
// tile w's stash (a stash copy is a few hundred bytes, so one CTA per tile
// would spend its life waiting on launch and load latency), then the whole
// CTA ranks the overflowing tiles among them one after another.
// ---------------------------------------------------------------------------
constexpr uint32_t kCompactTiles = kThreads / 32;

// Both schemes in one launch: the scheme is uniform per CTA (tiles of one tensor).
__global__ void __launch_bounds__(kThreads) compact_kernel(const __grid_constant__ EncBatch bt) {
  __shared__ uint32_t sm[kThreads / 32];
  __shared__ uint32_t overflow;
  const int ti = find_owner(bt, blockIdx.x);
  const EncDesc& d = bt.d[ti];
  const uint32_t t0 = (blockIdx.x - bt.prefix[ti]) * kCompactTiles;
  const uint32_t nt = min(kCompactTiles, d.n_tiles - t0);
  const uint32_t* tile_index = reinterpret_cast<const uint32_t*>(d.main + d.off_tile);
  uint32_t* pos = reinterpret_cast<uint32_t*>(d.esc + d.off_pos);
  uint16_t* val = reinterpret_cast<uint16_t*>(d.esc + d.off_val);
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) overflow = 0;
  __syncthreads();
  if (warp < nt) {
    const uint32_t t = t0 + warp;
    const uint32_t first = tile_index[t], count = tile_index[t + 1] - first;
    if (count > d.stash_cap) {
      if (lane == 0) atomicOr(&overflow, 1u << warp);
    } else {
      const uint64_t s0 = uint64_t(t) * d.stash_cap;
      // four entries per lane in flight before any is stored
      for (uint32_t i0 = 0; i0 < count; i0 += 128) {
        uint32_t p[4], v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t i = i0 + 32 * k + lane;
          if (i < count) {
            p[k] = d.stash_pos[s0 + i];
            v[k] = d.stash_val[s0 + i];
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t i = i0 + 32 * k + lane;
          if (i < count && first + i < d.E) {  // a count that disagrees with E is reported by the host
            pos[first + i] = p[k];
            val[first + i] = uint16_t(v[k]);
          }
        }
      }
    }
  }
  __syncthreads();
  const uint64_t G = cdiv(d.n, kGroup);
  for (uint32_t m = overflow; m; m &= m - 1) {  // uniform across the CTA
    const uint32_t t = t0 + uint32_t(__ffs(m) - 1);
    const uint64_t g = uint64_t(t) * kThreads + threadIdx.x;
    uint4 c4 = make_uint4(0, 0, 0, 0);
    if (g < G) c4 = *reinterpret_cast<const uint4*>(d.main + d.off_codes + 16 * g);
    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
    uint32_t cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = cw[i] & (cw[i] >> 1) & (cw[i] >> 2) & (cw[i] >> 3) & 0x11111111u;
      cnt += __popc(x);
    }
    uint32_t o = tile_index[t] + block_exclusive_256(cnt, sm);
    if (cnt) {
      const uint64_t base = g * kGroup;
      for (int e = 0; e < kGroup; ++e) {
        if (((cw[e >> 3] >> (4 * (e & 7))) & 0xF) == kEscape && o < d.E) {
          const uint32_t p = uint32_t(base + e);
          if (!WCOMP_DCHECK(p < d.n, 3)) break;
          pos[o] = p;
          val[o] = d.w[p];
          ++o;
        }
      }
    }
    __syncthreads();  // sm is rewritten by the next overflowing tile's scan
  }
}

// Row index: entry r = number of escapes below r * K (lower-bound search).
__global__ void __launch_bounds__(256) row_index_kernel(const __grid_constant__ EncBatch bt) {
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= bt.prefix[bt.count]) return;
  const int ti = find_owner(bt, x);
  const EncDesc& d = bt.d[ti];
  const int64_t r = int64_t(x - bt.prefix[ti]);
  const uint64_t bound = uint64_t(r) * uint64_t(d.K);
  const uint32_t* pos = reinterpret_cast<const uint32_t*>(d.esc + d.off_pos);
  uint64_t lo = 0, hi = d.E;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) >> 1;
    if (pos[mid] < bound) lo = mid + 1; else hi = mid;
  }
  reinterpret_cast<uint32_t*>(d.main + d.off_row)[r] = uint32_t(lo);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct Job {
  wcomp_container* c;
  EncDesc d;
};

// Histogram blocks for a tensor of n elements in a batch whose histogrammed
// tensors hold total_n elements: about 24 blocks per SM spread over the
// batch in proportion to size, but never fewer than keep every thread at or
// below kHistMaxChunks 8-element chunks (the 16-bit counter bound in
// hist_kernel), and never more than one chunk per thread.
uint32_t hist_blocks(uint64_t n, uint64_t total_n, int sms) {
  const uint64_t chunks = cdiv(n, 8);
  // about 24 blocks per SM over the launch, shared by tensor size (6 took
  // one layer's encode to 0.99 ms, 24 to 0.96 ms, 48 and 96 to 0.98 ms), but
  // at least 8 chunks a thread: a small tensor alone split thinner spends more
  // on its blocks' merges than it gains (2048 x 6144, both schemes: 0.105 ms
  // at 912 blocks, 0.123 ms at 3648)
  const uint64_t want = std::min<uint64_t>(std::max<uint64_t>(1, (uint64_t(sms) * 24 * n + total_n - 1) / total_n),
                                           cdiv(chunks, 8 * kHistThreads));
  const uint64_t need = cdiv(chunks, kHistMaxChunks * kHistThreads);
  return uint32_t(std::min<uint64_t>(std::max(want, need), cdiv(chunks, kHistThreads)));
}

void add_pad(ZeroList& z, uint8_t* base, uint64_t off, uint64_t sz) {
  const uint64_t p = padsec(sz);
  if (p == sz) return;
  z.p[z.count] = base + off + sz;
  z.len[z.count] = uint32_t(p - sz);
  ++z.count;
}

template <typename F>
cudaError_t for_chunks(std::vector<Job>& jobs, int scheme_filter, F&& launch) {
  std::vector<int> idx;
  for (int i = 0; i < int(jobs.size()); ++i)
    if (scheme_filter < 0 || jobs[i].d.scheme == scheme_filter) idx.push_back(i);
  for (size_t s = 0; s < idx.size(); s += kMaxBatch) {
    EncBatch b;
    memset(&b, 0, sizeof(b));
    b.count = int(std::min<size_t>(kMaxBatch, idx.size() - s));
    for (int j = 0; j < b.count; ++j) b.d[j] = jobs[idx[s + j]].d;
    launch(b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_zero(ZeroList& z, cudaStream_t s) {
  if (!z.count) return cudaSuccess;
  zero_kernel<<<z.count, 256, 0, s>>>(z);
  count_launches(1);
  z.count = 0;
  return cudaGetLastError();
}

// Escapes a tile's stash holds (pack records them, compaction copies them;
// a tile with more is ranked again from its codes).
constexpr uint32_t kStashCap = 512;

// Pinned host memory for one call's summaries, kept per host thread and
// grown on demand.  A call returns only after its copy into it completed.
Summary* pinned_summaries(int count) {
  thread_local Summary* buf = nullptr;
  thread_local int cap = 0;
  if (count > cap) {
    if (buf) cudaFreeHost(buf);
    buf = nullptr;
    cap = 0;
    if (cudaMallocHost(reinterpret_cast<void**>(&buf), sizeof(Summary) * size_t(count)) != cudaSuccess) {
      buf = nullptr;
      return nullptr;
    }
    cap = count;
  }
  return buf;
}

int encode_many(const uint16_t* const* ws, const int64_t* Ns, const int64_t* Ks, const int* schemes, int count,
                cudaStream_t s, wcomp_container** out) {
  for (int i = 0; i < count; ++i) out[i] = nullptr;
  for (int i = 0; i < count; ++i) {
    if (!ws[i] || Ns[i] <= 0 || Ks[i] <= 0) return WCOMP_EINVAL;
    if (schemes[i] != WCOMP_BYTESPLIT && schemes[i] != WCOMP_K15) return WCOMP_EINVAL;
    if (Ns[i] >= (int64_t(1) << 32) || Ks[i] >= (int64_t(1) << 32) ||
        uint64_t(Ns[i]) * uint64_t(Ks[i]) >= (uint64_t(1) << 32))
      return WCOMP_EUNSUPPORTED;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = sm_count(dev);
  std::vector<Job> jobs(count);
  for (auto& j : jobs) j.c = nullptr;
  Summary* d_sum = nullptr;
  auto fail = [&](cudaError_t err) -> int {
    for (auto& j : jobs)
      if (j.c) wcomp_free(j.c, s);
    if (d_sum) cudaFreeAsync(d_sum, s);
    return map_cuda(err);
  };
  cudaError_t e = pool_alloc(reinterpret_cast<void**>(&d_sum), sizeof(Summary) * count, s);
  if (e != cudaSuccess) return map_cuda(e);
  // the containers' main sections: one arena block for the whole batch, each
  // container's part starting on a 256-byte boundary
  Arena* main_arena = new (std::nothrow) Arena();
  if (!main_arena) return fail(cudaErrorMemoryAllocation);
  {
    uint64_t total = 0;
    for (int i = 0; i < count; ++i) {
      Layout L;
      L.compute(schemes[i], Ns[i], Ks[i], 0);
      total += (L.main_alloc + 255) & ~uint64_t(255);
    }
    e = pool_alloc(&main_arena->block, total, s);
    if (e != cudaSuccess) {
      delete main_arena;
      return fail(e);
    }
  }
  uint64_t main_off = 0;
  ZeroList z;
  memset(&z, 0, sizeof(z));
  for (int i = 0; i < count; ++i) {
    wcomp_container* c = new (std::nothrow) wcomp_container();
    if (!c) {
      if (main_arena->refs.load() == 0) {
        cudaFreeAsync(main_arena->block, s);
        delete main_arena;
      }
      return fail(cudaErrorMemoryAllocation);
    }
    jobs[i].c = c;
    c->device = dev;
    Layout& L = c->L;
    L.compute(schemes[i], Ns[i], Ks[i], 0);
    c->main_arena = main_arena;
    main_arena->refs.fetch_add(1, std::memory_order_relaxed);
    c->d_main = static_cast<uint8_t*>(main_arena->block) + main_off;
    main_off += (L.main_alloc + 255) & ~uint64_t(255);
    EncDesc& d = jobs[i].d;
    memset(&d, 0, sizeof(d));
    d.w = ws[i];
    d.main = c->d_main;
    d.summary = d_sum + i;
    d.n = L.n;
    d.N = L.N;
    d.K = L.K;
    d.off_codes = L.off_codes; d.off_raw = L.off_raw; d.off_a = L.off_a; d.off_b = L.off_b; d.off_c = L.off_c;
    d.off_tile = L.off_tile; d.off_row = L.off_row; d.off_scratch = L.off_scratch;
    d.n_tiles = uint32_t(L.n_tiles);
    d.scheme = schemes[i];
    d.aligned = (reinterpret_cast<uintptr_t>(ws[i]) & 15) == 0;
    z.p[z.count] = c->d_main + L.off_scratch + Scratch::hist;
    z.len[z.count] = kMaxBins * sizeof(uint32_t);
    ++z.count;
    // every section's padding up to its 32-byte boundary (pack's whole-group
    // stores cover only part of it for codes, raw bytes and plane A)
    add_pad(z, c->d_main, L.off_codes, L.sz_codes);
    add_pad(z, c->d_main, L.off_raw, L.sz_raw);
    add_pad(z, c->d_main, L.off_a, L.sz_a);
    add_pad(z, c->d_main, L.off_b, L.sz_b);
    add_pad(z, c->d_main, L.off_c, L.sz_c);
    add_pad(z, c->d_main, L.off_tile, L.sz_tile);
    add_pad(z, c->d_main, L.off_row, L.sz_row);
    if (z.count + 8 > kMaxZero && (e = launch_zero(z, s)) != cudaSuccess) return fail(e);
  }
  if ((e = launch_zero(z, s)) != cudaSuccess) return fail(e);

  // a1: histogram blocks in proportion to size, at most 8191 elements per thread
  // A byte-split job whose tensor is also encoded as K15 in this batch takes
  // its histogram from the K15 one instead of reading the source again.
  for (auto& j : jobs) j.d.hist_k15 = nullptr;
  for (auto& j : jobs) {
    if (j.d.scheme != WCOMP_BYTESPLIT) continue;
    for (auto& k : jobs)
      if (k.d.scheme == WCOMP_K15 && k.d.w == j.d.w && k.d.N == j.d.N && k.d.K == j.d.K) {
        j.d.hist_k15 = reinterpret_cast<const uint32_t*>(k.d.main + k.d.off_scratch + Scratch::hist);
        break;
      }
  }
  std::vector<Job> need_hist;
  for (auto& j : jobs)
    if (!j.d.hist_k15) need_hist.push_back(j);
  uint64_t total_n = 0;
  for (auto& j : jobs)
    if (!j.d.hist_k15) total_n += j.d.n;
  auto hist_launch = [&](int scheme) {
    return for_chunks(need_hist, scheme, [&](EncBatch& b) {
      uint32_t blocks = 0;
      for (int j = 0; j < b.count; ++j) {
        b.prefix[j] = blocks;
        blocks += hist_blocks(b.d[j].n, total_n, sms);
      }
      b.prefix[b.count] = blocks;
      if (scheme == WCOMP_BYTESPLIT)
        hist_kernel<8, 256><<<blocks, 256, 0, s>>>(b);
      else
        hist_kernel<7, 512><<<blocks, 256, 0, s>>>(b);
      count_launches(1);
    });
  };
  auto tiles_prefix = [](EncBatch& b) {
    uint32_t t = 0;
    for (int j = 0; j < b.count; ++j) {
      b.prefix[j] = t;
      t += b.d[j].n_tiles;
    }
    b.prefix[b.count] = t;
    return t;
  };
  if ((e = hist_launch(WCOMP_BYTESPLIT)) != cudaSuccess) return fail(e);
  if ((e = hist_launch(WCOMP_K15)) != cudaSuccess) return fail(e);
  // a2: tables, and E from the histogram (n minus the table symbols' counts)
  e = for_chunks(jobs, -1, [&](EncBatch& b) {
    select_kernel<<<b.count, 512, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail(e);

  // Pack does not need E: its stash holds a fixed number of escapes per
  // tile (a tile with more is ranked again by the compaction), so pack and
  // the tile scan are queued before the host waits for E, and the wait (on
  // an event after the summaries' copy, not on the stream) overlaps them.
  uint64_t stash_entries = 0;
  for (int i = 0; i < count; ++i) stash_entries += uint64_t(kStashCap) * jobs[i].c->L.n_tiles;
  uint8_t* stash = nullptr;
  e = pool_alloc(reinterpret_cast<void**>(&stash), stash_entries * 6, s);
  if (e != cudaSuccess) return fail(e);
  {
    uint64_t off = 0;
    for (int i = 0; i < count; ++i) {
      jobs[i].d.stash_cap = kStashCap;
      jobs[i].d.stash_pos = reinterpret_cast<uint32_t*>(stash) + off;
      jobs[i].d.stash_val = reinterpret_cast<uint16_t*>(stash + 4 * stash_entries) + off;
      off += uint64_t(kStashCap) * jobs[i].c->L.n_tiles;
    }
  }
  auto fail2 = [&](cudaError_t err) -> int {
    if (stash) cudaFreeAsync(stash, s);
    return fail(err);
  };
  // escape counts and tables to pinned host memory, then the event the host
  // waits on; the second half of the buffer receives the summaries again
  // after the tile scan (the escapes actually found)
  Summary* hs = pinned_summaries(2 * count);
  if (!hs) return fail2(cudaErrorMemoryAllocation);
  Summary* hs2 = hs + count;
  cudaEvent_t ready = nullptr, scanned = nullptr;
  e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&scanned, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemcpyAsync(hs, d_sum, sizeof(Summary) * count, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaEventRecord(ready, s);
  if (e != cudaSuccess) {
    if (ready) cudaEventDestroy(ready);
    if (scanned) cudaEventDestroy(scanned);
    return fail2(e);
  }
  // past this point copies into the pinned buffer may be in flight: wait for them before leaving
  bool scanned_recorded = false;
  auto drain = [&]() {
    cudaEventSynchronize(ready);
    cudaEventDestroy(ready);
    ready = nullptr;
    if (scanned_recorded) cudaEventSynchronize(scanned);
    cudaEventDestroy(scanned);
    scanned = nullptr;
  };
  auto fail3 = [&](cudaError_t err) -> int {
    drain();
    return fail2(err);
  };
  // a3: pack (with the stash), then the tile scan.  A byte-split job and a
  // K15 job of the same tensor are packed together, reading the source once.
  std::vector<Job> pairs, singles;  // pairs: byte-split, K15, byte-split, K15, ...
  {
    std::vector<char> paired(jobs.size(), 0);
    for (size_t j = 0; j < jobs.size(); ++j) {
      if (jobs[j].d.scheme != WCOMP_BYTESPLIT) continue;
      for (size_t k = 0; k < jobs.size(); ++k)
        if (!paired[k] && jobs[k].d.scheme == WCOMP_K15 && jobs[k].d.w == jobs[j].d.w &&
            jobs[k].d.N == jobs[j].d.N && jobs[k].d.K == jobs[j].d.K) {
          paired[j] = paired[k] = 1;
          pairs.push_back(jobs[j]);
          pairs.push_back(jobs[k]);
          break;
        }
    }
    for (size_t j = 0; j < jobs.size(); ++j)
      if (!paired[j]) singles.push_back(jobs[j]);
  }
  for (size_t s0 = 0; s0 < pairs.size(); s0 += kMaxBatch) {
    EncBatch b;
    memset(&b, 0, sizeof(b));
    b.count = int(std::min<size_t>(kMaxBatch, pairs.size() - s0));
    uint32_t t = 0;
    for (int j = 0; j < b.count; ++j) b.d[j] = pairs[s0 + j].d;
    for (int i = 0; i < b.count / 2; ++i) {
      b.prefix[i] = t;
      t += b.d[2 * i].n_tiles;
    }
    b.prefix[b.count / 2] = t;
    pack_twin_kernel<<<t, kThreads, 0, s>>>(b);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail3(e);
  }
  e = for_chunks(singles, WCOMP_BYTESPLIT, [&](EncBatch& b) {
    pack_kernel<WCOMP_BYTESPLIT><<<tiles_prefix(b), kThreads, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail3(e);
  e = for_chunks(singles, WCOMP_K15, [&](EncBatch& b) {
    pack_kernel<WCOMP_K15><<<tiles_prefix(b), kThreads, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail3(e);
  e = for_chunks(jobs, -1, [&](EncBatch& b) {
    scan_kernel<<<b.count, 1024, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail3(e);
  e = cudaMemcpyAsync(hs2, d_sum, sizeof(Summary) * count, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaEventRecord(scanned, s);
  if (e != cudaSuccess) return fail3(e);
  scanned_recorded = true;
  cudaFreeAsync(d_sum, s);
  d_sum = nullptr;
  // first wait: escape counts and tables (pack and the scan keep running)
  e = cudaEventSynchronize(ready);
  if (e != cudaSuccess) return fail3(e);
  // the escape streams, sized now that E is known: one arena block for the batch
  uint64_t esc_total = 0;
  for (int i = 0; i < count; ++i) {
    Layout L = jobs[i].c->L;
    L.compute(L.scheme, L.N, L.K, hs[i].E);
    if (L.E) esc_total += (L.esc_alloc + 255) & ~uint64_t(255);
  }
  Arena* esc_arena = nullptr;
  if (esc_total) {
    esc_arena = new (std::nothrow) Arena();
    if (!esc_arena) return fail3(cudaErrorMemoryAllocation);
    e = pool_alloc(&esc_arena->block, esc_total, s);
    if (e != cudaSuccess) {
      delete esc_arena;
      return fail3(e);
    }
  }
  uint64_t esc_off = 0;
  for (int i = 0; i < count; ++i) {
    wcomp_container* c = jobs[i].c;
    memcpy(c->table, hs[i].table, sizeof(c->table));
    Layout& L = c->L;
    L.compute(L.scheme, L.N, L.K, hs[i].E);
    EncDesc& d = jobs[i].d;
    d.E = L.E;
    d.off_pos = L.off_pos;
    d.off_val = L.off_val;
    if (L.E) {
      c->esc_arena = esc_arena;
      esc_arena->refs.fetch_add(1, std::memory_order_relaxed);
      c->d_esc = static_cast<uint8_t*>(esc_arena->block) + esc_off;
      esc_off += (L.esc_alloc + 255) & ~uint64_t(255);
      d.esc = c->d_esc;
      add_pad(z, c->d_esc, L.off_pos, L.sz_pos);
      add_pad(z, c->d_esc, L.off_val, 2 * L.E);
      if (z.count + 2 > kMaxZero && (e = launch_zero(z, s)) != cudaSuccess) return fail3(e);
    }
  }
  if ((e = launch_zero(z, s)) != cudaSuccess) return fail3(e);
  // a4: compaction for tensors with escapes; row indexes for all
  std::vector<Job> with_esc;
  for (auto& j : jobs)
    if (j.d.E) with_esc.push_back(j);
  e = for_chunks(with_esc, -1, [&](EncBatch& b) {
    uint32_t blocks = 0;
    for (int j = 0; j < b.count; ++j) {
      b.prefix[j] = blocks;
      blocks += uint32_t(cdiv(b.d[j].n_tiles, kCompactTiles));
    }
    b.prefix[b.count] = blocks;
    compact_kernel<<<blocks, kThreads, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail3(e);
  e = for_chunks(jobs, -1, [&](EncBatch& b) {
    uint32_t rows = 0;
    for (int j = 0; j < b.count; ++j) {
      b.prefix[j] = rows;
      rows += uint32_t(b.d[j].N + 1);
    }
    b.prefix[b.count] = rows;
    row_index_kernel<<<unsigned(cdiv(rows, 256)), 256, 0, s>>>(b);
    count_launches(1);
  });
  if (e != cudaSuccess) return fail3(e);
  if (stash) cudaFreeAsync(stash, s);
  stash = nullptr;
  // second wait, for the tile scan (the compaction and the row indexes queued
  // above keep running): the escapes pack found must number the E the
  // histogram implied, which sized the escape streams.  A mismatch means a
  // wrong histogram; the compaction wrote nothing past E, and no container is
  // returned.
  e = cudaEventSynchronize(scanned);
  drain();
  if (e != cudaSuccess) return fail2(e);
  for (int i = 0; i < count; ++i)
    if (hs2[i].scanned != hs[i].E) {
      for (auto& j : jobs)
        if (j.c) wcomp_free(j.c, s);
      return WCOMP_EINTERNAL;
    }
  for (int i = 0; i < count; ++i) out[i] = jobs[i].c;
  return WCOMP_OK;
}

}  // namespace

WCOMP_DEBUG_TAKE(debug_take_encode)
}  // namespace wc

using namespace wc;

extern "C" int wcomp_encode(const uint16_t* d_w, int64_t N, int64_t K, int scheme, void* stream,
                            wcomp_container** out) {
  if (!out) return WCOMP_EINVAL;
  *out = nullptr;
  if (!d_w || N <= 0 || K <= 0) return WCOMP_EINVAL;
  return encode_many(&d_w, &N, &K, &scheme, 1, static_cast<cudaStream_t>(stream), out);
}

extern "C" int wcomp_encode_hist_grid(const uint64_t* n, int count, int sms, uint32_t* blocks) {
  if (!n || !blocks || count <= 0 || sms <= 0) return WCOMP_EINVAL;
  uint64_t total_n = 0;
  for (int i = 0; i < count; ++i) {
    if (n[i] == 0 || n[i] >= (uint64_t(1) << 32)) return WCOMP_EINVAL;
    total_n += n[i];
  }
  for (int i = 0; i < count; ++i) blocks[i] = hist_blocks(n[i], total_n, sms);
  return WCOMP_OK;
}

extern "C" int wcomp_encode_batched(const uint16_t* const* d_w, const int64_t* N, const int64_t* K,
                                    const int* schemes, int count, void* stream, wcomp_container** out) {
  if (!d_w || !N || !K || !schemes || !out || count <= 0) return WCOMP_EINVAL;
  return encode_many(d_w, N, K, schemes, count, static_cast<cudaStream_t>(stream), out);
}
