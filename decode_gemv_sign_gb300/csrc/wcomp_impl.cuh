// Internal definitions shared by the library's translation units: the
// container object, the device layout of its streams, kernel descriptors and
// the register-level decode helpers.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is reached through the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/wcomp.h"

namespace wc {

constexpr int kTableSize = 15;
constexpr int kEscape = 15;
constexpr uint32_t kTile = 8192;   // elements per decode tile / tile-index granule
constexpr int kGroup = 32;         // elements per thread group (one K15 plane group)
constexpr int kHeaderBytes = 96;
constexpr int kMaxBins = 512;

__host__ __device__ inline uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline uint64_t padsec(uint64_t x) { return (x + 31) & ~uint64_t(31); }  // section alignment: 32 bytes

// Byte offsets of every stream.  "main" holds the sections whose size is known
// before encoding (codes, raw or planes, indexes) followed by encoder scratch;
// "esc" holds the escape positions and values, sized once E is known.
struct Layout {
  int scheme;
  int64_t N, K;
  uint64_t n, groups, n_tiles, E;
  // sizes (unpadded) and offsets within main / esc
  uint64_t sz_codes, sz_raw, sz_a, sz_b, sz_c, sz_tile, sz_row, sz_pos, sz_val;
  uint64_t off_codes, off_raw, off_a, off_b, off_c, off_tile, off_row;
  uint64_t main_payload;   // serialized bytes of the main sections
  uint64_t off_scratch;    // encoder scratch (not serialized)
  uint64_t main_alloc;
  uint64_t off_pos, off_val, esc_payload;
  // On the device every escape value is the whole 16-bit word (byte-split's
  // low byte repeats the raw byte), so no kernel re-reads the raw stream for
  // an escape; the serialized form keeps byte-split values as the high byte.
  uint64_t esc_alloc;

  void compute(int scheme_, int64_t N_, int64_t K_, uint64_t E_) {
    scheme = scheme_;
    N = N_;
    K = K_;
    n = uint64_t(N) * uint64_t(K);
    groups = cdiv(n, kGroup);
    n_tiles = cdiv(n, kTile);
    E = E_;
    sz_codes = cdiv(n, 2);
    sz_raw = scheme == WCOMP_BYTESPLIT ? n : 0;
    sz_a = scheme == WCOMP_K15 ? 16 * groups : 0;
    sz_b = scheme == WCOMP_K15 ? 8 * groups : 0;
    sz_c = scheme == WCOMP_K15 ? 4 * groups : 0;
    sz_tile = 4 * (n_tiles + 1);
    sz_row = 4 * (uint64_t(N) + 1);
    sz_pos = 4 * E;
    sz_val = scheme == WCOMP_BYTESPLIT ? E : 2 * E;
    uint64_t o = 0;
    off_codes = o; o += padsec(sz_codes);
    off_raw = o; o += padsec(sz_raw);
    off_a = o; o += padsec(sz_a);
    off_b = o; o += padsec(sz_b);
    off_c = o; o += padsec(sz_c);
    off_tile = o; o += padsec(sz_tile);
    off_row = o; o += padsec(sz_row);
    main_payload = o;
    off_scratch = o;
    main_alloc = o + 4096;
    off_pos = 0;
    off_val = padsec(sz_pos);
    esc_payload = padsec(sz_pos) + padsec(sz_val);
    esc_alloc = padsec(sz_pos) + padsec(2 * E);
  }
  uint64_t serialized() const { return kHeaderBytes + main_payload + esc_payload; }
};

// Encoder scratch inside the main allocation.
struct Scratch {
  static constexpr uint64_t hist = 0;          // uint32[512]
  static constexpr uint64_t lut = 2048;        // uint8[512]: symbol -> code
  static constexpr uint64_t table = 2560;      // uint16[16]: code -> symbol (16th = 0)
};

}  // namespace wc

namespace wc {
// Device memory shared by the containers of one batched encode (one block for
// their main sections, one for their escape streams): returned to the pool
// when the last container using it is released.
struct Arena {
  void* block = nullptr;
  std::atomic<int> refs{0};
};
}  // namespace wc

struct wcomp_container {
  wc::Layout L;
  uint16_t table[wc::kTableSize];
  uint8_t* d_main = nullptr;       // inside main_arena when that is set, else its own allocation
  uint8_t* d_esc = nullptr;        // inside esc_arena when that is set, else its own allocation
  wc::Arena* main_arena = nullptr;
  wc::Arena* esc_arena = nullptr;
  int device = 0;
  // TMA descriptors of the code and raw / mantissa streams, made on the
  // first fused GEMV (tmap_ok: 1 made, 0 not applicable to this shape)
  CUtensorMap tmap[4];
  int tmap_ok = 0;
  std::once_flag tmap_once;
};

namespace wc {

// The register form of the 16-entry code table: the high bytes of the 15
// symbols plus the placeholder 0 for code 15, four per 32-bit word, and for
// K15 the exponent LSB of each symbol as 0x80 / 0x00 bytes.
struct RegTable {
  uint32_t hi[4];
  uint32_t e0[4];
};

inline RegTable make_reg_table(const uint16_t* table, int scheme) {
  RegTable t{};
  for (int c = 0; c < 16; ++c) {
    uint32_t s = c < kTableSize ? table[c] : 0u;  // placeholder symbol 0 for the escape code
    uint32_t hi = scheme == WCOMP_BYTESPLIT ? (s & 0xFF) : ((s >> 1) & 0xFF);
    uint32_t e0 = scheme == WCOMP_BYTESPLIT ? 0u : ((s & 1u) ? 0x80u : 0u);
    t.hi[c >> 2] |= hi << (8 * (c & 3));
    t.e0[c >> 2] |= e0 << (8 * (c & 3));
  }
  return t;
}

// One tensor as seen by the decode and GEMV kernels.
struct TensorDesc {
  const uint8_t* codes;
  const uint8_t* raw;      // byte-split low bytes
  const uint8_t* pa;       // K15 planes
  const uint8_t* pb;
  const uint8_t* pc;
  const uint32_t* tile_index;
  const uint32_t* row_index;
  const uint32_t* esc_pos;
  const uint16_t* esc_val;  // whole 16-bit words of the escaped elements
  uint64_t n;
  uint64_t E;              // escapes
  int64_t N, K;
  RegTable t;
  int scheme;
  int aligned;             // streams and output 32-byte aligned: vector path allowed
};

inline TensorDesc make_desc(const wcomp_container* c) {
  const Layout& L = c->L;
  TensorDesc d{};
  d.codes = c->d_main + L.off_codes;
  d.raw = c->d_main + L.off_raw;
  d.pa = c->d_main + L.off_a;
  d.pb = c->d_main + L.off_b;
  d.pc = c->d_main + L.off_c;
  d.tile_index = reinterpret_cast<const uint32_t*>(c->d_main + L.off_tile);
  d.row_index = reinterpret_cast<const uint32_t*>(c->d_main + L.off_row);
  d.esc_pos = reinterpret_cast<const uint32_t*>(c->d_esc + L.off_pos);
  d.esc_val = reinterpret_cast<const uint16_t*>(c->d_esc + L.off_val);
  d.n = L.n;
  d.E = L.E;
  d.N = L.N;
  d.K = L.K;
  d.t = make_reg_table(c->table, L.scheme);
  d.scheme = L.scheme;
  d.aligned = 1;
  return d;
}

// Batched launches carry their descriptors as a kernel parameter.
constexpr int kMaxBatch = 32;

struct DecodeBatch {
  TensorDesc d[kMaxBatch];
  uint16_t* out[kMaxBatch];
  uint32_t tile_prefix[kMaxBatch + 1];  // first global tile of each tensor
  int count;
};

struct GemvBatch {
  TensorDesc d[kMaxBatch];
  const uint16_t* x[kMaxBatch];
  float* y[kMaxBatch];
  uint32_t set_prefix[kMaxBatch + 1];   // first global row set of each tensor
  int count;
  uint64_t l2_bytes;                    // the device's L2 size (sizes the escape prefetch)
};

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t lop_select(uint32_t lo, uint32_t hi, uint32_t m) {
  // (lo & ~m) | (hi & m)
  return (lo & ~m) | (hi & m);
}

// Table bytes for the 8 codes of one 32-bit code word: returns the bytes of
// elements 0..3 in *q0 and 4..7 in *q1.  `m7` is the word masked with
// 0x77777777 (the 3-bit in-half index of every code).
struct QuadMasks {
  uint32_t m0, m1;  // 0xFF bytes where the code is >= 8
};

__device__ __forceinline__ QuadMasks code_masks(uint32_t cw) {
  // prmt in sign-replicate mode copies bit 7 of the picked byte to all 8 bits;
  // bit 3 of nibble j sits at bit 7 of byte j/2 of (cw << 4) (j even) or cw (j odd).
  uint32_t s = cw << 4;
  QuadMasks m;
  m.m0 = prmt(s, cw, 0xD9C8);
  m.m1 = prmt(s, cw, 0xFBEA);
  return m;
}

__device__ __forceinline__ void lookup8(const uint32_t* t4, uint32_t m7, const QuadMasks& m,
                                        uint32_t& q0, uint32_t& q1) {
  uint32_t h = m7 >> 16;
  q0 = lop_select(prmt(t4[0], t4[1], m7), prmt(t4[2], t4[3], m7), m.m0);
  q1 = lop_select(prmt(t4[0], t4[1], h), prmt(t4[2], t4[3], h), m.m1);
}

// K15 mantissas.  A 32-element group keeps its 7-bit mantissas in 28 bytes,
// seen as seven 32-bit words W0..W6 (W0..W3 in plane A, W4..W5 in plane B,
// W6 in plane C): byte lane i of W_q holds element 4q + i in bits 0..6, and
// its bit 7 holds bit q of the mantissa of element 28 + i.  Quad q < 7 is
// therefore W_q with bit 7 cleared; quad 7 gathers bit 7 of every word.
__device__ __forceinline__ uint32_t k15_tail(const uint32_t (&w)[7]) {
  uint32_t r = 0;
#pragma unroll
  for (int q = 0; q < 7; ++q) r |= (w[q] >> (7 - q)) & (0x01010101u << q);
  return r;
}

// Decode one 32-element group into 16 words of BF16 pairs (element 2j in the
// low half of word j).  Escaped elements carry the placeholder (symbol 0).
template <int SCHEME>
__device__ __forceinline__ void decode_group(const RegTable& t, const uint32_t (&cw)[4],
                                             const uint32_t (&r)[8], uint32_t (&out)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    QuadMasks m = code_masks(cw[i]);
    uint32_t m7 = cw[i] & 0x77777777u;
    uint32_t h0, h1;
    lookup8(t.hi, m7, m, h0, h1);
    uint32_t l0, l1;
    if (SCHEME == WCOMP_BYTESPLIT) {
      l0 = r[2 * i];
      l1 = r[2 * i + 1];
    } else {
      uint32_t e0, e1;
      lookup8(t.e0, m7, m, e0, e1);
      l0 = r[2 * i] | e0;
      l1 = r[2 * i + 1] | e1;
    }
    out[4 * i + 0] = prmt(l0, h0, 0x5140);
    out[4 * i + 1] = prmt(l0, h0, 0x7362);
    out[4 * i + 2] = prmt(l1, h1, 0x5140);
    out[4 * i + 3] = prmt(l1, h1, 0x7362);
  }
}

// K15: the 8 mantissa quads of a group from its plane words (bit 7 of every
// byte cleared; the exponent bit is added by the caller).
__device__ __forceinline__ void k15_mantissas(const uint32_t (&a)[4], const uint32_t (&b)[2], uint32_t c,
                                              uint32_t (&r)[8]) {
  const uint32_t w[7] = {a[0], a[1], a[2], a[3], b[0], b[1], c};
#pragma unroll
  for (int q = 0; q < 7; ++q) r[q] = w[q] & 0x7F7F7F7Fu;
  r[7] = k15_tail(w);
}

// Streaming loads that do not keep the weights in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void ld_stream_v8(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st_v8(void* p, const uint32_t* r) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Load the code words and raw words of group g (vector path, full group).
template <int SCHEME>
__device__ __forceinline__ void load_group(const TensorDesc& d, uint64_t g, uint32_t (&cw)[4],
                                           uint32_t (&r)[8]) {
  uint4 c4 = ld_stream_v4(d.codes + 16 * g);
  cw[0] = c4.x; cw[1] = c4.y; cw[2] = c4.z; cw[3] = c4.w;
  if (SCHEME == WCOMP_BYTESPLIT) {
    ld_stream_v8(d.raw + 32 * g, r);
  } else {
    uint4 a4 = ld_stream_v4(d.pa + 16 * g);
    uint2 b2 = ld_stream_v2(d.pb + 8 * g);
    uint32_t c = ld_stream_u32(d.pc + 4 * g);
    uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
    uint32_t b[2] = {b2.x, b2.y};
    k15_mantissas(a, b, c, r);
  }
}

// Byte j (0..27) of the mantissa bytes of group g: plane A bytes 0..15,
// plane B bytes 16..23, plane C bytes 24..27.
__device__ __forceinline__ uint32_t k15_mant_byte(const TensorDesc& d, uint64_t g, uint32_t j) {
  return j < 16 ? d.pa[16 * g + j] : j < 24 ? d.pb[8 * g + (j - 16)] : d.pc[4 * g + (j - 24)];
}

// The 7-bit mantissa of element i.
__device__ __forceinline__ uint32_t k15_mant_elem(const TensorDesc& d, uint64_t i) {
  const uint64_t g = i >> 5;
  const uint32_t e = uint32_t(i & 31);
  if (e < 28) return k15_mant_byte(d, g, e) & 0x7F;
  uint32_t m = 0;
  for (uint32_t q = 0; q < 7; ++q) m |= ((k15_mant_byte(d, g, 4 * q + (e - 28)) >> 7) & 1u) << q;
  return m;
}

// Element-wise decode of element i (any alignment; escapes give the placeholder).
__device__ __forceinline__ uint32_t decode_elem_placeholder(const TensorDesc& d, uint64_t i) {
  uint32_t code = (d.codes[i >> 1] >> (4 * (i & 1))) & 0xF;
  uint32_t hi = (d.t.hi[code >> 2] >> (8 * (code & 3))) & 0xFF;
  uint32_t lo;
  if (d.scheme == WCOMP_BYTESPLIT) {
    lo = d.raw[i];
  } else {
    uint32_t e0 = (d.t.e0[code >> 2] >> (8 * (code & 3))) & 0x80;
    lo = e0 | k15_mant_elem(d, i);
  }
  return (hi << 8) | lo;
}


__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Shared-memory address of a generic pointer into shared memory.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// Debug builds (WCOMP_DEBUG=1): index checks before the kernels' memory
// accesses.  A failed check sets a bit in the translation unit's error word
// and the access is skipped, so the kernel finishes; wcomp_device_check
// reports it as WCOMP_EBOUNDS.  Release builds compile the checks away.
//   bit 0: decode output or escape position out of range
//   bit 1: GEMV escape position, row or column out of range
//   bit 2: GEMV output or x index out of range
//   bit 3: encoder stash or escape stream index out of range
// ---------------------------------------------------------------------------
#ifndef WCOMP_DEBUG
#define WCOMP_DEBUG 0
#endif
#if WCOMP_DEBUG
#define WCOMP_DEBUG_WORD static __device__ uint32_t g_debug_err;
#define WCOMP_DCHECK(cond, bit) ((cond) ? true : (atomicOr(&g_debug_err, 1u << (bit)), false))
#define WCOMP_DEBUG_TAKE(fn)                                                          \
  uint32_t fn() {                                                                     \
    uint32_t v = 0, z = 0;                                                            \
    if (cudaMemcpyFromSymbol(&v, g_debug_err, sizeof(v)) != cudaSuccess) return ~0u; \
    cudaMemcpyToSymbol(g_debug_err, &z, sizeof(z));                                   \
    return v;                                                                         \
  }
#else
#define WCOMP_DEBUG_WORD
#define WCOMP_DCHECK(cond, bit) true
#define WCOMP_DEBUG_TAKE(fn) \
  uint32_t fn() { return 0; }
#endif
// Each translation unit's debug error word, read and cleared (0 in release builds).
uint32_t debug_take_decode();
uint32_t debug_take_encode();
uint32_t debug_take_gemv();

// Host-side launch helpers (defined in container.cu).
// Stream-ordered allocation from the library's own memory pool on the current
// device (created on first use; it keeps freed blocks for reuse instead of
// returning them to the driver at every synchronization).
cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s);
int sm_count(int device);
uint64_t l2_size(int device);
int map_cuda(cudaError_t e);
void count_launches(uint64_t k);

}  // namespace wc
