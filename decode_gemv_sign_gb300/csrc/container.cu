// Container life cycle on the host: info, serialization (header + CRC-32),
// validation of serialized bytes, upload, release, status strings.
//
// The pages define no file format: both serialized forms are this library's
// own.  The compact form (version 2) stores what the forgeeks page "Prueba de
// GLM-5.2 reduce la memoria BF16 en casi un 25%" counts in its bits per weight
// (section "Cómo funciona la compresión"): codes, raw bits, and each escape at
// its symbol width, its position implied by its code 15.  Every byte handed to
// wcomp_deserialize is checked on the host before it reaches the device, the
// corruption checks the wavect page "Compresión de pesos LLM sin pérdida vs
// 8-bit GGUF" asks of a production pilot (section "Un piloto de producción de
// 14 días").
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "wcomp_impl.cuh"

namespace wc {

int map_cuda(cudaError_t e) {
  if (e == cudaSuccess) return WCOMP_OK;
  if (e == cudaErrorMemoryAllocation) return WCOMP_ENOMEM;
  return WCOMP_ECUDA;
}

static std::atomic<uint64_t> g_launches{0};
void count_launches(uint64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s) {
  static std::mutex mu;
  static cudaMemPool_t pools[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!pools[dev]) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t pool;
      e = cudaMemPoolCreate(&pool, &props);
      if (e != cudaSuccess) return e;
      uint64_t keep = ~uint64_t(0);
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      pools[dev] = pool;
    }
  }
  return cudaMallocFromPoolAsync(p, bytes, pools[dev], s);
}

int sm_count(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> g(mu);
  if (device < 0 || device >= 64) return 148;
  if (!cache[device]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) v = 148;
    cache[device] = v;
  }
  return cache[device];
}

uint64_t l2_size(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> g(mu);
  if (device < 0 || device >= 64) return 0;
  if (!cache[device]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, device) != cudaSuccess || v <= 0) v = -1;
    cache[device] = v;
  }
  return cache[device] > 0 ? uint64_t(cache[device]) : 0;
}

// CRC-32 (IEEE 802.3 polynomial, reflected, initial value and final xor 0xFFFFFFFF).
static uint32_t crc_table[256];
static std::once_flag crc_once;

static void crc_init() {
  for (uint32_t i = 0; i < 256; ++i) {
    uint32_t c = i;
    for (int k = 0; k < 8; ++k) c = (c & 1) ? (0xEDB88320u ^ (c >> 1)) : (c >> 1);
    crc_table[i] = c;
  }
}

uint32_t crc32_update(uint32_t crc, const uint8_t* p, size_t len) {
  std::call_once(crc_once, crc_init);
  crc = ~crc;
  for (size_t i = 0; i < len; ++i) crc = crc_table[(crc ^ p[i]) & 0xFF] ^ (crc >> 8);
  return ~crc;
}

static void put16(uint8_t* p, uint16_t v) { memcpy(p, &v, 2); }
static void put32(uint8_t* p, uint32_t v) { memcpy(p, &v, 4); }
static void put64(uint8_t* p, uint64_t v) { memcpy(p, &v, 8); }
static uint16_t get16(const uint8_t* p) { uint16_t v; memcpy(&v, p, 2); return v; }
static uint32_t get32(const uint8_t* p) { uint32_t v; memcpy(&v, p, 4); return v; }
static uint64_t get64(const uint8_t* p) { uint64_t v; memcpy(&v, p, 8); return v; }

}  // namespace wc

using namespace wc;

extern "C" int wcomp_version(void) { return WCOMP_VERSION; }

extern "C" uint64_t wcomp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char* wcomp_strerror(int s) {
  switch (s) {
    case WCOMP_OK: return "ok";
    case WCOMP_EINVAL: return "invalid argument";
    case WCOMP_ENOMEM: return "out of memory";
    case WCOMP_ECORRUPT: return "corrupt container";
    case WCOMP_ECUDA: return "CUDA error";
    case WCOMP_EUNSUPPORTED: return "unsupported size";
    case WCOMP_ETIMEOUT: return "a device wait timed out";
    case WCOMP_EINTERNAL: return "internal consistency check failed";
    case WCOMP_EBOUNDS: return "a kernel index check failed (debug build)";
    default: return "unknown status";
  }
}

// The compact serialized form (format version 2).  Its codes and raw bytes /
// K15 planes keep their version-1 offsets (they lead both forms); then one
// u16 escape count per tile and the escape symbols (u8, or 9 bits packed
// least significant bit first for K15).  Positions, the row index and the
// K15 escape mantissas are rebuilt from the codes and planes when loading.
constexpr uint16_t kVersionCompact = 2;

struct CompactLayout {
  uint64_t sz_tilecount, sz_sym, off_tilecount, off_sym, payload;
  void compute(const Layout& L) {
    sz_tilecount = 2 * L.n_tiles;
    sz_sym = L.scheme == WCOMP_BYTESPLIT ? L.E : cdiv(9 * L.E, 8);
    off_tilecount = L.off_tile;
    off_sym = off_tilecount + padsec(sz_tilecount);
    payload = off_sym + padsec(sz_sym);
  }
  uint64_t serialized() const { return kHeaderBytes + payload; }
};

extern "C" int wcomp_info(const wcomp_container* c, wcomp_info_t* info) {
  if (!c || !info) return WCOMP_EINVAL;
  const Layout& L = c->L;
  memset(info, 0, sizeof(*info));
  info->scheme = L.scheme;
  info->version = WCOMP_VERSION;
  info->N = L.N;
  info->K = L.K;
  info->n = int64_t(L.n);
  info->n_escapes = L.E;
  info->tile_elems = kTile;
  info->n_tiles = uint32_t(L.n_tiles);
  for (int i = 0; i < kTableSize; ++i) info->table[i] = c->table[i];
  info->bytes_codes = padsec(L.sz_codes);
  info->bytes_raw = padsec(L.sz_raw) + padsec(L.sz_a) + padsec(L.sz_b) + padsec(L.sz_c);
  info->bytes_index = padsec(L.sz_tile) + padsec(L.sz_row);
  info->bytes_escapes = L.esc_payload;
  info->serialized_bytes = L.serialized();
  const double sym_bits = L.scheme == WCOMP_BYTESPLIT ? 8.0 : 9.0;
  const double raw_bits = L.scheme == WCOMP_BYTESPLIT ? 8.0 : 7.0;
  info->entropy_bpw = 4.0 + raw_bits + (double(L.E) + kTableSize) * sym_bits / double(L.n);
  info->physical_bpw = 8.0 * double(L.serialized()) / double(L.n);
  CompactLayout C;
  C.compute(L);
  info->serialized_compact_bytes = C.serialized();
  info->physical_compact_bpw = 8.0 * double(C.serialized()) / double(L.n);
  return WCOMP_OK;
}

static void write_header(const wcomp_container* c, uint16_t version, uint64_t payload_len, uint32_t payload_crc,
                         uint8_t* h) {
  const Layout& L = c->L;
  memset(h, 0, kHeaderBytes);
  memcpy(h, "WCMP", 4);
  put16(h + 4, version);
  h[6] = uint8_t(L.scheme);
  put64(h + 8, uint64_t(L.N));
  put64(h + 16, uint64_t(L.K));
  put64(h + 24, L.E);
  put32(h + 32, kTile);
  for (int i = 0; i < kTableSize; ++i) put16(h + 40 + 2 * i, c->table[i]);
  put64(h + 72, payload_len);
  put32(h + 80, payload_crc);
  put32(h + 92, crc32_update(0, h, 92));
}

extern "C" int wcomp_serialize(const wcomp_container* c, void* host_buf, uint64_t cap, uint64_t* len,
                               void* stream) {
  if (!c || !len) return WCOMP_EINVAL;
  const Layout& L = c->L;
  *len = L.serialized();
  if (!host_buf) return WCOMP_OK;
  if (cap < L.serialized()) return WCOMP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* out = static_cast<uint8_t*>(host_buf);
  uint8_t* esc = out + kHeaderBytes + L.main_payload;
  // the device keeps whole escape words; version 1 stores byte-split values
  // as the high byte
  std::vector<uint16_t> words(L.scheme == WCOMP_BYTESPLIT ? L.E : 0);
  cudaError_t e = cudaMemcpyAsync(out + kHeaderBytes, c->d_main, L.main_payload, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && L.E) {
    memset(esc, 0, L.esc_payload);
    e = cudaMemcpyAsync(esc + L.off_pos, c->d_esc + L.off_pos, L.sz_pos, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = L.scheme == WCOMP_BYTESPLIT
              ? cudaMemcpyAsync(words.data(), c->d_esc + L.off_val, 2 * L.E, cudaMemcpyDeviceToHost, s)
              : cudaMemcpyAsync(esc + L.off_val, c->d_esc + L.off_val, L.sz_val, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return map_cuda(e);
  for (uint64_t r = 0; r < words.size(); ++r) esc[L.off_val + r] = uint8_t(words[r] >> 8);
  uint32_t crc = crc32_update(0, out + kHeaderBytes, L.main_payload + L.esc_payload);
  write_header(c, WCOMP_VERSION, L.main_payload + L.esc_payload, crc, out);
  return WCOMP_OK;
}

extern "C" int wcomp_serialize_compact(const wcomp_container* c, void* host_buf, uint64_t cap, uint64_t* len,
                                       void* stream) {
  if (!c || !len) return WCOMP_EINVAL;
  const Layout& L = c->L;
  CompactLayout C;
  C.compute(L);
  *len = C.serialized();
  if (!host_buf) return WCOMP_OK;
  if (cap < C.serialized()) return WCOMP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* out = static_cast<uint8_t*>(host_buf);
  uint8_t* p = out + kHeaderBytes;
  std::vector<uint32_t> tile(L.n_tiles + 1);
  std::vector<uint16_t> val(L.E);  // whole escape words
  // codes and raw bytes / planes in one copy (same offsets in both forms)
  cudaError_t e = cudaMemcpyAsync(p, c->d_main, L.off_tile, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(tile.data(), c->d_main + L.off_tile, L.sz_tile, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && L.E)
    e = cudaMemcpyAsync(val.data(), c->d_esc + L.off_val, 2 * L.E, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return map_cuda(e);
  uint8_t* tc = p + C.off_tilecount;
  memset(tc, 0, padsec(C.sz_tilecount));
  for (uint64_t t = 0; t < L.n_tiles; ++t) put16(tc + 2 * t, uint16_t(tile[t + 1] - tile[t]));
  uint8_t* sym = p + C.off_sym;
  memset(sym, 0, padsec(C.sz_sym));
  if (L.scheme == WCOMP_BYTESPLIT) {
    for (uint64_t r = 0; r < L.E; ++r) sym[r] = uint8_t(val[r] >> 8);  // the high byte
  } else {
    for (uint64_t r = 0; r < L.E; ++r) {
      const uint32_t v = uint32_t(val[r]) >> 7;  // the 9-bit symbol
      const uint64_t bit = 9 * r;
      const uint32_t w = v << (bit & 7);
      sym[bit >> 3] |= uint8_t(w);
      sym[(bit >> 3) + 1] |= uint8_t(w >> 8);
    }
  }
  const uint32_t crc = crc32_update(0, p, C.payload);
  write_header(c, kVersionCompact, C.payload, crc, out);
  return WCOMP_OK;
}

// Host-side validation of a serialized container (nothing reaches the device
// unless every check passes, so the kernels never see out-of-range positions).
// Header fields shared by both forms: magic, header checksum, version,
// scheme, sizes, tile size and the table (15 distinct symbols in range).
// Fills L for the container's shape and returns the format version.
static int check_header(const uint8_t* b, uint64_t len, Layout& L, uint16_t* table, uint16_t* version) {
  if (len < uint64_t(kHeaderBytes)) return WCOMP_ECORRUPT;
  if (memcmp(b, "WCMP", 4) != 0) return WCOMP_ECORRUPT;
  if (get32(b + 92) != crc32_update(0, b, 92)) return WCOMP_ECORRUPT;
  *version = get16(b + 4);
  if (*version != WCOMP_VERSION && *version != kVersionCompact) return WCOMP_ECORRUPT;
  int scheme = b[6];
  if (scheme != WCOMP_BYTESPLIT && scheme != WCOMP_K15) return WCOMP_ECORRUPT;
  int64_t N = int64_t(get64(b + 8)), K = int64_t(get64(b + 16));
  uint64_t E = get64(b + 24);
  if (get32(b + 32) != kTile) return WCOMP_ECORRUPT;
  if (N <= 0 || K <= 0 || N > (int64_t(1) << 32) || K > (int64_t(1) << 32)) return WCOMP_ECORRUPT;
  uint64_t n = uint64_t(N) * uint64_t(K);
  if (n >= (uint64_t(1) << 32) || E > n) return WCOMP_ECORRUPT;
  L.compute(scheme, N, K, E);
  const int nb = scheme == WCOMP_BYTESPLIT ? 256 : 512;
  for (int i = 0; i < kTableSize; ++i) {
    table[i] = get16(b + 40 + 2 * i);
    if (table[i] >= nb) return WCOMP_ECORRUPT;
    for (int j = 0; j < i; ++j)
      if (table[j] == table[i]) return WCOMP_ECORRUPT;
  }
  return WCOMP_OK;
}

static int validate(const uint8_t* b, uint64_t len, const Layout& L) {
  const int64_t N = L.N, K = L.K;
  const uint64_t n = L.n, E = L.E;
  if (get64(b + 72) != L.main_payload + L.esc_payload) return WCOMP_ECORRUPT;
  if (len != L.serialized()) return WCOMP_ECORRUPT;
  const uint8_t* p = b + kHeaderBytes;
  if (get32(b + 80) != crc32_update(0, p, L.main_payload + L.esc_payload)) return WCOMP_ECORRUPT;
  // escape positions: strictly ascending, below n, exactly the elements coded 15
  const uint8_t* codes = p + L.off_codes;
  const uint8_t* pos = p + L.main_payload + L.off_pos;
  uint64_t e = 0;
  for (uint64_t i = 0; i < n; ++i) {
    uint32_t code = (codes[i >> 1] >> (4 * (i & 1))) & 0xF;
    if (code == kEscape) {
      if (e >= E || get32(pos + 4 * e) != i) return WCOMP_ECORRUPT;
      ++e;
    }
  }
  if (e != E) return WCOMP_ECORRUPT;
  // tile and row indexes: escapes below each boundary
  const uint8_t* ti = p + L.off_tile;
  uint64_t k = 0;
  for (uint64_t t = 0; t <= L.n_tiles; ++t) {
    uint64_t bound = t * kTile;
    while (k < E && get32(pos + 4 * k) < bound) ++k;
    if (get32(ti + 4 * t) != k) return WCOMP_ECORRUPT;
  }
  const uint8_t* ri = p + L.off_row;
  k = 0;
  for (uint64_t r = 0; r <= uint64_t(N); ++r) {
    uint64_t bound = r * uint64_t(K);
    while (k < E && get32(pos + 4 * k) < bound) ++k;
    if (get32(ri + 4 * r) != k) return WCOMP_ECORRUPT;
  }
  return WCOMP_OK;
}

// K15 mantissa of element i.  A 32-element group keeps 28 mantissa bytes: 16
// in plane A, 8 in plane B, 4 in plane C.  Byte j < 28 holds element j in
// bits 0..6; bit 7 of byte 4 q + l holds bit q of element 28 + l.
static uint32_t k15_mantissa(const uint8_t* pa, const uint8_t* pb, const uint8_t* pc, uint64_t i) {
  const uint64_t g = i >> 5;
  const uint32_t e = uint32_t(i & 31);
  auto byte_at = [&](uint32_t j) -> uint32_t {
    return j < 16 ? pa[16 * g + j] : j < 24 ? pb[8 * g + (j - 16)] : pc[4 * g + (j - 24)];
  };
  if (e < 28) return byte_at(e) & 0x7Fu;
  uint32_t m = 0;
  for (uint32_t q = 0; q < 7; ++q) m |= ((byte_at(4 * q + (e - 28)) >> 7) & 1u) << q;
  return m;
}

// Compact form: check the payload and rebuild the version-1 sections
// (positions from the codes 15, tile and row indexes, whole K15 escape
// words) into main / esc images laid out like a version-1 payload.
static int load_compact(const uint8_t* b, uint64_t len, const Layout& L, std::vector<uint8_t>& main_img,
                        std::vector<uint8_t>& esc_img) {
  CompactLayout C;
  C.compute(L);
  if (get64(b + 72) != C.payload || len != C.serialized()) return WCOMP_ECORRUPT;
  const uint8_t* p = b + kHeaderBytes;
  if (get32(b + 80) != crc32_update(0, p, C.payload)) return WCOMP_ECORRUPT;
  main_img.assign(L.main_payload, 0);
  esc_img.assign(L.esc_payload, 0);
  memcpy(main_img.data(), p, L.off_tile);  // codes and raw bytes / planes
  const uint8_t* codes = p + L.off_codes;
  const uint8_t* tc = p + C.off_tilecount;
  uint8_t* pos = esc_img.data() + L.off_pos;
  uint8_t* ti = main_img.data() + L.off_tile;
  // positions: the elements coded 15, in order; E of them, matching every tile count
  uint64_t e = 0;
  for (uint64_t t = 0; t < L.n_tiles; ++t) {
    put32(ti + 4 * t, uint32_t(e));
    const uint64_t lo = t * kTile, hi = lo + kTile < L.n ? lo + kTile : L.n;
    const uint64_t e0 = e;
    for (uint64_t i = lo; i < hi; ++i) {
      if (((codes[i >> 1] >> (4 * (i & 1))) & 0xF) != kEscape) continue;
      if (e >= L.E) return WCOMP_ECORRUPT;
      put32(pos + 4 * e, uint32_t(i));
      ++e;
    }
    if (e - e0 != get16(tc + 2 * t)) return WCOMP_ECORRUPT;
  }
  if (e != L.E) return WCOMP_ECORRUPT;
  put32(ti + 4 * L.n_tiles, uint32_t(e));
  uint8_t* ri = main_img.data() + L.off_row;
  uint64_t k = 0;
  for (uint64_t r = 0; r <= uint64_t(L.N); ++r) {
    const uint64_t bound = r * uint64_t(L.K);
    while (k < L.E && get32(pos + 4 * k) < bound) ++k;
    put32(ri + 4 * r, uint32_t(k));
  }
  const uint8_t* sym = p + C.off_sym;
  uint8_t* val = esc_img.data() + L.off_val;
  if (L.scheme == WCOMP_BYTESPLIT) {
    if (L.E) memcpy(val, sym, L.E);
  } else {
    for (uint64_t r = 0; r < L.E; ++r) {
      const uint64_t bit = 9 * r;
      const uint32_t v = ((uint32_t(sym[bit >> 3]) | (uint32_t(sym[(bit >> 3) + 1]) << 8)) >> (bit & 7)) & 0x1FFu;
      const uint32_t m = k15_mantissa(p + L.off_a, p + L.off_b, p + L.off_c, get32(pos + 4 * r));
      put16(val + 2 * r, uint16_t((v << 7) | m));
    }
  }
  return WCOMP_OK;
}

extern "C" int wcomp_deserialize(const void* host_buf, uint64_t len, void* stream, wcomp_container** out) {
  if (!host_buf || !out) return WCOMP_EINVAL;
  *out = nullptr;
  const uint8_t* b = static_cast<const uint8_t*>(host_buf);
  Layout L;
  uint16_t table[kTableSize];
  uint16_t version = 0;
  int st = check_header(b, len, L, table, &version);
  if (st != WCOMP_OK) return st;
  std::vector<uint8_t> main_img, esc_img;
  const uint8_t* main_src = b + kHeaderBytes;
  const uint8_t* esc_src = main_src + L.main_payload;
  if (version == WCOMP_VERSION) {
    st = validate(b, len, L);
  } else {
    st = load_compact(b, len, L, main_img, esc_img);
    main_src = main_img.data();
    esc_src = esc_img.data();
  }
  if (st != WCOMP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wcomp_container* c = new (std::nothrow) wcomp_container();
  if (!c) return WCOMP_ENOMEM;
  c->L = L;
  memcpy(c->table, table, sizeof(table));
  cudaGetDevice(&c->device);
  // the device escape section: positions, then whole 16-bit words (a
  // byte-split value joins its high byte with the element's raw low byte)
  std::vector<uint8_t> dev_esc(L.E ? L.esc_alloc : 0, 0);
  if (L.E) {
    memcpy(dev_esc.data() + L.off_pos, esc_src + L.off_pos, L.sz_pos);
    uint8_t* w = dev_esc.data() + L.off_val;
    const uint8_t* v = esc_src + L.off_val;
    if (L.scheme == WCOMP_BYTESPLIT) {
      const uint8_t* raw = main_src + L.off_raw;
      for (uint64_t r = 0; r < L.E; ++r) put16(w + 2 * r, uint16_t((uint32_t(v[r]) << 8) | raw[get32(esc_src + L.off_pos + 4 * r)]));
    } else {
      memcpy(w, v, 2 * L.E);
    }
  }
  cudaError_t e = pool_alloc(reinterpret_cast<void**>(&c->d_main), L.main_alloc, s);
  if (e == cudaSuccess && L.E) e = pool_alloc(reinterpret_cast<void**>(&c->d_esc), L.esc_alloc, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->d_main, main_src, L.main_payload, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && L.E)
    e = cudaMemcpyAsync(c->d_esc, dev_esc.data(), L.esc_alloc, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    wcomp_free(c, stream);
    return map_cuda(e);
  }
  *out = c;
  return WCOMP_OK;
}

// Release one container's hold on a block: its own allocation, or its share
// of an arena (the arena's block goes back to the pool with the last share).
static void release_block(Arena* a, void* own, cudaStream_t s) {
  if (a) {
    if (a->refs.fetch_sub(1, std::memory_order_acq_rel) == 1) {
      cudaFreeAsync(a->block, s);
      delete a;
    }
  } else if (own) {
    cudaFreeAsync(own, s);
  }
}

extern "C" void wcomp_free(wcomp_container* c, void* stream) {
  if (!c) return;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  release_block(c->main_arena, c->d_main, s);
  release_block(c->esc_arena, c->d_esc, s);
  delete c;
}
