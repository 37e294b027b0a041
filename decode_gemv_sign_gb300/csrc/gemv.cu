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
// One kernel covers every batch size and every source (byte-split, K15, plain
// BF16).  The product runs on the tensor cores with warp-level
// mma.sync.m16n8k16 (BF16 in, fp32 accumulate): the rebuilt weights are the
// MMA's A operand (16 weight rows by 16 columns), x is the B operand (16
// columns by 8 batch rows; a second MMA on the same A covers batch rows 8..15).
// The multiply is never the bound; moving the compressed bytes is.
//
// Work unit: 16 consecutive rows of one tensor.  A CTA of 8 warps takes a unit
// and splits its K range into 8 runs of 128-column k-blocks; the warps' 16 x 8
// (or 16 x 16) partial tiles are summed in shared memory in a fixed order.
// CTA i starts on unit i and takes further units from a global counter, so
// tensors of any shape share one launch; a launch with one CTA per unit (up
// to two units per resident CTA slot) leaves the counter alone.  K15 with the
// transposed x, and the plain GEMV above B = 8, walk each run from an offset
// that depends on the unit (runs of 16 k-blocks or more), so the CTAs do not
// all read the same x lines at once.
//
// Lane (g = lane / 4, t = lane % 4) of a warp owns rows g and g + 8 of the
// unit and, in every k-block, the 32 columns 32 t .. 32 t + 31: one whole
// 32-element group of each row (16 bytes of codes plus 32 raw bytes, or plus
// the 28 K15 mantissa bytes, or 64 bytes of plain BF16).  The MMA's column
// order inside a step is a relabelling shared by the weights and x (column
// slot 2t + j of step s is column 32 t + 4 s + j of the k-block), which leaves
// the sum unchanged.
//
// Bytes in flight.  Every warp owns a ring of kStages shared-memory stages.
// One lane brings k-block kb of the unit's 16 rows into a stage with one 2-D
// tensor copy (TMA, cp.async.bulk.tensor) per stream: a box of 16 rows by 64
// bytes of codes and 128 raw bytes (K15: 64, 32 and 16 bytes of mantissa
// planes; plain: two boxes of 128 bytes), kStages - 1 k-blocks ahead of the
// one the warp computes and across unit boundaries, completing on the
// stage's mbarrier.  Raw and plain boxes land 128-byte swizzled, so the
// lanes' 16-byte reads of a stage are free of bank conflicts.  Waits are
// bounded: a stage that never completes sets the device error word and the
// warp stops waiting (its results are then undefined), drains what it has in
// flight and finishes, so no launch can hang.
//
// Escapes.  An escaped weight decodes to the placeholder (symbol 0, so
// |w| < 2^-125); threads add x * (w_true - w_placeholder) over the unit's
// escapes (found in O(1) through the row index), moved through the k-loop in
// a three-stage register pipeline and finished at the unit's end, and the
// parts are summed in a fixed order.  For K15 at B >= 3 the corrections read
// a copy of x transposed to [K][4, 8 or 16], made by a pre-pass, so one
// thread takes every batch row of an escape at once.
// Results never depend on which warp ran which unit: no atomics touch the
// sums.
#include <string.h>

#include <algorithm>
#include <atomic>
#include <memory>
#include <mutex>
#include <new>
#include <vector>

#include "wcomp_impl.cuh"

namespace wc {
namespace {
WCOMP_DEBUG_WORD
#if WCOMP_DEBUG
// Debug builds: when set, every warp of a GEMV launch leaves its first copy
// unissued but waits for it, so that bounded wait runs out.
__device__ uint32_t g_debug_skip_first_copy;
#endif

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlots = 1024;   // work-counter slots per device (one per launch, round robin)
constexpr int kRows = 16;      // weight rows per unit (the MMA's M side)
constexpr int kKBlock = 128;   // columns per k-block (4 lanes x 32)
constexpr int kCtasPerSm = 2;
constexpr int kEscDepth = 16;  // escape corrections with their loads in flight together

enum Src { kBytesplit = WCOMP_BYTESPLIT, kK15 = WCOMP_K15, kPlain = 2 };

// Copies of the code-pair table per instantiation (0: register lookups).
// K15 needs two table bytes per element (the high byte and the exponent bit),
// so at B <= 4 one shared-memory lookup per code byte beats two register
// lookups; sixteen copies, one per lane residue mod 16, leave only lanes l and
// l + 16 able to collide on a bank (measured on a 16384 x 53248 weight: 8 -> 16
// copies cut B = 1 from 332 to 317 us and B = 16 from 600 to 568 us; 32
// copies, 32 KB a CTA, took L1 from the corrections and were slower at B = 16).
// Above B = 4 the transposed-x gathers of the corrections want that L1 more
// than the decode wants the table: register lookups took B = 8 from 408 to
// 403 us and B = 16 from 539 to 523 us (and B = 1 from 305 to 350 us, B = 2
// from 363 to 367 us, so the table stays there).  Byte-split needs only the
// high byte and decodes from registers.
template <int SRC, int NT, int XW>
constexpr int lut_rep() { return SRC == kK15 && NT == 1 && XW <= 4 ? 16 : 0; }

// Escapes a correction thread moves one stage along per k-block, and the most
// stages a warp's ring keeps, per instantiation (XW: width of the transposed
// x, 0 = none).  K15 up to 8 batch rows moves one aligned quad (4 entries);
// the others move single entries.  Measured on a 16384 x 53248 weight: K15,
// with 3 % escapes, gains from deeper in-loop corrections (B = 1: 2 -> 4 cut
// 385 to 347 us, and quads with vector loads instead of four single entries
// 316 to 310 us; B = 3..8 with the transposed x: 1 -> 2 cut 483 to 400 us at
// B = 4, and quads 422 -> 408 us at B = 8) and from
// two stages, whose smaller shared-memory share leaves more L1 to the
// corrections and to x (three stages: B = 1 305 -> 313 us, B = 16 569 -> 666
// us); with two batch tiles (NT = 2) deeper corrections spill registers.
// Byte-split with two batch tiles also keeps two stages (against three: B = 9
// 277 -> 272 us, B = 16 322 -> 318 us).
template <int SRC, int NT, int XW>
constexpr int esc_q() { return SRC != kK15 ? 2 : XW <= 8 ? 4 : 1; }
template <int SRC, int NT>
constexpr int max_stages() { return SRC == kK15 || (SRC == kBytesplit && NT == 2) ? 2 : 4; }

// One stage of one warp in shared memory, as the tensor copies write it (row
// r of a box at r times its row length; regions start on 1024-byte
// boundaries, which the 128-byte swizzle needs):
//   byte-split: codes [16][64] at 0, raw bytes [16][128] (swizzled) at 1024
//   K15:        codes [16][64] at 0, plane A [16][64] at 1024, plane B [16][32]
//               at 2048, plane C [16][16] at 2560
//   plain:      columns 0..63 [16][128 bytes] (swizzled) at 0, 64..127 at 2048
template <int SRC>
struct StageGeom {
  static constexpr uint32_t kTx = SRC == kBytesplit ? 3072 : SRC == kK15 ? 2816 : 4096;  // bytes per k-block
  static constexpr uint32_t kBytes = (kTx + 1023) & ~1023u;
};

// 128-byte swizzle of a box with 128-byte rows: the 16-byte chunk c of row r
// sits at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ int owner(const uint32_t* prefix, int count, uint32_t u, int start = 0) {
  int i = start;
  while (i + 1 < count && prefix[i + 1] <= u) ++i;
  return i;
}

__device__ __forceinline__ uint32_t load_esc_val(const TensorDesc& d, uint32_t e) { return d.esc_val[e]; }

// w_true - w_placeholder for one escape whose whole word is `val`: the
// placeholder keeps the element's own low bits (byte-split: the raw low byte;
// K15: the 7-bit mantissa) under symbol 0.
template <int SCHEME>
__device__ __forceinline__ float esc_delta(uint32_t val) {
  const uint32_t wph = val & (SCHEME == WCOMP_BYTESPLIT ? 0xFFu : 0x7Fu);
  return __uint_as_float(val << 16) - __uint_as_float(wph << 16);
}

// The same for the two escapes whose whole words are the halves of w.
template <int SCHEME>
__device__ __forceinline__ void esc_delta_pair(uint32_t w, float& d_lo, float& d_hi) {
  constexpr uint32_t lm = SCHEME == WCOMP_BYTESPLIT ? 0xFFu : 0x7Fu;
  d_lo = __uint_as_float(w << 16) - __uint_as_float((w & lm) << 16);
  d_hi = __uint_as_float(w & 0xFFFF0000u) - __uint_as_float(w & (lm << 16));
}

// 32 bytes of x (one column of the 16-wide transposed x) in one load: one
// request per escape instead of two (measured on a 16384 x 53248 weight: K15
// B = 16 568 -> 537 us, B = 9 508 -> 496 us).
__device__ __forceinline__ void ld_x_v8(const uint16_t* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

__device__ __forceinline__ uint4 ld_x_v4(const uint16_t* p) {
  uint4 v;
  asm("ld.global.nc.L1::evict_last.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// TMA and mbarriers.
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitNs = 1000000000ull;  // how long a wait on a stage's copies may take (1 s)

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t x, uint32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_init_u32(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_done(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of the given parity; false if it has not completed by
// `deadline` (global timer, ns).
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_done(bar, parity))
    if (global_ns() > deadline) return false;
  return true;
}
// The same with a deadline kWaitNs from the first poll that failed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  return mbar_done(bar, parity) || mbar_wait_until(bar, parity, global_ns() + kWaitNs);
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Tensor maps of one launch: for tensor i, map 0 is the code stream (or the
// plain BF16 rows), maps 1..3 the raw bytes or the K15 planes A, B, C.  Each
// views its stream as a 2-D array of N rows of bytes.
struct TmaBatch {
  CUtensorMap m[kMaxBatch][4];
};

// ---------------------------------------------------------------------------
// A unit and this warp's share of it.
// ---------------------------------------------------------------------------
struct Unit {
  int ti;
  int64_t r0;
  int rows;            // valid rows (1..16)
  uint32_t kb0, kb1;   // this warp's k-blocks [kb0, kb1)
  uint32_t kvalid;     // valid columns of the tensor's last k-block (32..128)
  uint32_t nkb;        // k-blocks per row
  uint32_t rot;        // the warp walks [kb0, kb1) from kb0 + rot, wrapping around
};

// rot_mul: 0 (every warp walks its k-range in order), or the factor that
// spreads the starting offsets of successive units over ranges of at least 16
// k-blocks, where the walk was measured to gain (16384 x 53248 and 6144 x
// 16384, K15 B = 4: 364 -> 331 and 65.1 -> 63.0 us); on six k-blocks a warp
// (K = 6144) it made no difference either way.
__device__ __forceinline__ void unit_of(const GemvBatch& p, uint32_t u, int start, int warp, Unit& m,
                                        uint32_t rot_mul) {
  m.ti = owner(p.set_prefix, p.count, u, start);
  const TensorDesc& d = p.d[m.ti];
  m.r0 = int64_t(u - p.set_prefix[m.ti]) * kRows;
  m.rows = int(d.N - m.r0 < kRows ? d.N - m.r0 : kRows);
  m.nkb = uint32_t(cdiv(uint64_t(d.K), kKBlock));
  m.kvalid = uint32_t(d.K - int64_t(m.nkb - 1) * kKBlock);
  m.kb0 = uint32_t(uint64_t(m.nkb) * warp / kWarps);
  m.kb1 = uint32_t(uint64_t(m.nkb) * (warp + 1) / kWarps);
  const uint32_t span = m.kb1 - m.kb0;
  m.rot = span >= 16 ? uint32_t(uint64_t(u) * rot_mul % span) : 0u;
}

// The i-th k-block (kb0 <= i < kb1) in the warp's walk of unit m.
__device__ __forceinline__ uint32_t kb_at(const Unit& m, uint32_t i) {
  const uint32_t a = i + m.rot;
  return a >= m.kb1 ? a - (m.kb1 - m.kb0) : a;
}

// Bring k-block kb of unit m into the stage at `st` (one lane of the warp):
// rows past N and columns past K arrive as zeros.
template <int SRC>
__device__ __forceinline__ void issue_item(const TmaBatch& tm, const Unit& m, uint32_t kb, uint32_t st, uint32_t bar) {
  const CUtensorMap* mp = tm.m[m.ti];
  const uint32_t y = uint32_t(m.r0);
  mbar_arrive_tx(bar, StageGeom<SRC>::kTx);
  if (SRC == kPlain) {
    tma_load_2d(st, mp, kb * 256, y, bar);
    tma_load_2d(st + 2048, mp, kb * 256 + 128, y, bar);
  } else {
    tma_load_2d(st, mp, kb * 64, y, bar);
    if (SRC == kBytesplit) {
      tma_load_2d(st + 1024, mp + 1, kb * 128, y, bar);
    } else {
      tma_load_2d(st + 1024, mp + 1, kb * 64, y, bar);
      tma_load_2d(st + 2048, mp + 2, kb * 32, y, bar);
      tma_load_2d(st + 2560, mp + 3, kb * 16, y, bar);
    }
  }
}

// BF16 pairs of one code word (8 elements): P[j] holds elements 2j, 2j+1.
// l0 / l1 are the low bytes of elements 0..3 / 4..7 (byte-split: raw bytes;
// K15: mantissa bytes with bit 7 cleared).
template <int SRC>
__device__ __forceinline__ void pairs8(const RegTable& tab, uint32_t cw, uint32_t l0, uint32_t l1,
                                       uint32_t (&P)[4]) {
  const QuadMasks m = code_masks(cw);
  const uint32_t m7 = cw & 0x77777777u;
  uint32_t h0, h1;
  lookup8(tab.hi, m7, m, h0, h1);
  if (SRC == kK15) {
    uint32_t e0, e1;
    lookup8(tab.e0, m7, m, e0, e1);
    l0 |= e0;
    l1 |= e1;
  }
  P[0] = prmt(l0, h0, 0x5140);
  P[1] = prmt(l0, h0, 0x7362);
  P[2] = prmt(l1, h1, 0x5140);
  P[3] = prmt(l1, h1, 0x7362);
}

// The same pairs from the shared-memory code-pair table: entry v (a code
// byte: the codes of two consecutive elements) holds, as bytes, the K15
// exponent bit (bit 7) and high byte of the low nibble's symbol, then those of
// the high nibble's symbol (byte-split: 0, symbol, 0, symbol).  lut is this
// lane's copy (lut_rep copies interleaved word by word, lane % lut_rep).
template <int SRC, int REP>
__device__ __forceinline__ void pairs8_lut(uint32_t lut, uint32_t cw, uint32_t l0, uint32_t l1, uint32_t (&P)[4]) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t v = prmt(cw, 0u, 0x4440u + b);
    const uint32_t T = lds32(lut + v * (REP * 4));
    const uint32_t w = prmt(b < 2 ? l0 : l1, T, (b & 1) ? 0x7352u : 0x7150u);
    P[b] = SRC == kK15 ? ((w & ~0x00800080u) | (T & 0x00800080u)) : w;
  }
}

// One k-block of this lane from its stage: decode the two groups code word
// by code word and issue the MMAs (two per code word and batch tile).  In a
// k-block that ends past K (FULL false) a lane whose columns are all past K
// (live false) feeds zero weights: its zero-filled codes would decode to the
// table's first symbol, which need not be finite.
template <int SRC, int NT, bool FULL, int REP>
__device__ __forceinline__ void compute_item(const RegTable& tab, uint32_t lut, uint32_t st, int lane, bool live,
                                             const uint4 (&xv)[NT][4], float (&acc)[NT][4]) {
  const uint32_t g = uint32_t(lane) >> 2, t = uint32_t(lane) & 3;
  uint32_t cg[4], ch[4], lg[8], lh[8];
  if (SRC == kPlain) {
    // row g columns 32 t .. +31 are 16-byte chunks 4 (t & 1) + i of the box t / 2
    const uint32_t half = st + (t >> 1) * 2048;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t c = 4 * (t & 1) + i;
      const uint4 wg = lds128(half + swz(g, c)), wh = lds128(half + swz(g + 8, c));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16(acc[nt], wg.x, wh.x, wg.y, wh.y, xv[nt][i].x, xv[nt][i].y);
        mma_bf16(acc[nt], wg.z, wh.z, wg.w, wh.w, xv[nt][i].z, xv[nt][i].w);
      }
    }
    return;
  }
  {
    const uint4 c0 = lds128(st + g * 64 + t * 16), c1 = lds128(st + (g + 8) * 64 + t * 16);
    cg[0] = c0.x; cg[1] = c0.y; cg[2] = c0.z; cg[3] = c0.w;
    ch[0] = c1.x; ch[1] = c1.y; ch[2] = c1.z; ch[3] = c1.w;
  }
  if (SRC == kBytesplit) {
    const uint32_t r = st + 1024;
    const uint4 r0 = lds128(r + swz(g, 2 * t)), r1 = lds128(r + swz(g, 2 * t + 1));
    const uint4 r2 = lds128(r + swz(g + 8, 2 * t)), r3 = lds128(r + swz(g + 8, 2 * t + 1));
    lg[0] = r0.x; lg[1] = r0.y; lg[2] = r0.z; lg[3] = r0.w; lg[4] = r1.x; lg[5] = r1.y; lg[6] = r1.z; lg[7] = r1.w;
    lh[0] = r2.x; lh[1] = r2.y; lh[2] = r2.z; lh[3] = r2.w; lh[4] = r3.x; lh[5] = r3.y; lh[6] = r3.z; lh[7] = r3.w;
  } else {
    const uint4 ag = lds128(st + 1024 + g * 64 + t * 16), ah = lds128(st + 1024 + (g + 8) * 64 + t * 16);
    const uint2 bg = lds64(st + 2048 + g * 32 + t * 8), bh = lds64(st + 2048 + (g + 8) * 32 + t * 8);
    const uint32_t cgw = lds32(st + 2560 + g * 16 + t * 4), chw = lds32(st + 2560 + (g + 8) * 16 + t * 4);
    const uint32_t wg[7] = {ag.x, ag.y, ag.z, ag.w, bg.x, bg.y, cgw};
    const uint32_t wh[7] = {ah.x, ah.y, ah.z, ah.w, bh.x, bh.y, chw};
    // bit 7 of every byte carries a tail-element bit: cleared here for the
    // register lookups, replaced by the exponent bit in the table lookups
#pragma unroll
    for (int q = 0; q < 7; ++q) {
      lg[q] = REP ? wg[q] : wg[q] & 0x7F7F7F7Fu;
      lh[q] = REP ? wh[q] : wh[q] & 0x7F7F7F7Fu;
    }
    lg[7] = k15_tail(wg);
    lh[7] = k15_tail(wh);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t P[4], H[4];
    if (REP) {
      pairs8_lut<SRC, REP>(lut, cg[i], lg[2 * i], lg[2 * i + 1], P);
      pairs8_lut<SRC, REP>(lut, ch[i], lh[2 * i], lh[2 * i + 1], H);
    } else {
      pairs8<SRC>(tab, cg[i], lg[2 * i], lg[2 * i + 1], P);
      pairs8<SRC>(tab, ch[i], lh[2 * i], lh[2 * i + 1], H);
    }
    if (!FULL && !live) {
#pragma unroll
      for (int q = 0; q < 4; ++q) P[q] = H[q] = 0u;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_bf16(acc[nt], P[0], H[0], P[1], H[1], xv[nt][i].x, xv[nt][i].y);
      mma_bf16(acc[nt], P[2], H[2], P[3], H[3], xv[nt][i].z, xv[nt][i].w);
    }
  }
}

// x of k-block kb for this lane: batch rows g (and g + 8 when NT == 2),
// columns 32 t .. 32 t + 31; zeros for batch rows >= B and columns past K.
// With PF, the 128-byte lines of the same columns of k-block kb + 1 are
// prefetched into L1, so the next call finds them there (measured on a
// 16384 x 53248 weight: byte-split B = 4 289 -> 238 us, plain 283 -> 268 us,
// K15 B = 1 310 -> 306 us; K15 with the transposed x and two batch tiles gain
// nothing).
template <int NT, bool PF>
__device__ __forceinline__ void load_x(const GemvBatch& p, const Unit& m, uint32_t kb, int B, int lane,
                                       uint4 (&xv)[NT][4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t valid = kb + 1 == m.nkb ? m.kvalid : uint32_t(kKBlock);
  const bool kok = uint32_t(32 * t) < valid;
  const int64_t K = p.d[m.ti].K;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int b = g + 8 * nt;
    if (kok && b < B && WCOMP_DCHECK(int64_t(kb) * kKBlock + 32 * t + 32 <= K, 2)) {
      const uint16_t* xr = p.x[m.ti] + int64_t(b) * K + int64_t(kb) * kKBlock + 32 * t;
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[nt][i] = ld_x_v4(xr + 8 * i);
      if (PF && (t & 1) == 0 && int64_t(kb + 1) * kKBlock + 32 * t + 64 <= K)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(xr + kKBlock));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[nt][i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// x transposed for the escape corrections: xt[i][k * XW + b] = x_i[b, k]
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
  static_assert(XW == 4 || XW == 8 || XW == 16, "transposed width");
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
    if (XW == 4) {
      *reinterpret_cast<uint2*>(out) = make_uint2(v[0], v[1 % (XW / 2)]);
    } else {
#pragma unroll
      for (int q = 0; q < XW / 8; ++q)
        reinterpret_cast<uint4*>(out)[q] = make_uint4(v[(4 * q) % (XW / 2)], v[(4 * q + 1) % (XW / 2)],
                                                      v[(4 * q + 2) % (XW / 2)], v[(4 * q + 3) % (XW / 2)]);
    }
  }
}

// Shared memory of one CTA (dynamic): the warps' stage rings, the stages'
// mbarriers, partial tiles, escape corrections and the unit hand-over words,
// plus room to round the base up to 1024 bytes.  Each warp keeps as many
// stages (2 to 4) as let two CTAs share an SM.
constexpr uint32_t kSmemPerCta = 112 * 1024;

template <int SRC, int NT, int XW, int ST>
struct SmemAt {
  static constexpr uint32_t kRing = kWarps * ST * StageGeom<SRC>::kBytes;
  static constexpr uint32_t kBarOff = kRing;
  static constexpr uint32_t kPartOff = kBarOff + kWarps * ST * 8;
  static constexpr uint32_t kPart = 2 * kWarps * 32 * 4 * NT;                        // floats
  static constexpr uint32_t kCorr = SRC == kPlain ? 0 : XW > 0 ? 2 * kRows * 16 : 2 * kThreads;  // floats
  static constexpr uint32_t kCorrOff = kPartOff + 4 * kPart;
  static constexpr uint32_t kLutOff = kCorrOff + 4 * kCorr;
  static constexpr uint32_t kLut = 256 * lut_rep<SRC, NT, XW>();  // words
  static constexpr uint32_t kUnitOff = kLutOff + 4 * kLut;  // first unit, next unit x 2
  static constexpr uint32_t kBytes = kUnitOff + 16 + 1024;
};

template <int SRC, int NT, int XW>
constexpr int ring_stages() {
  return max_stages<SRC, NT>() >= 4 && SmemAt<SRC, NT, XW, 4>::kBytes <= kSmemPerCta   ? 4
         : max_stages<SRC, NT>() >= 3 && SmemAt<SRC, NT, XW, 3>::kBytes <= kSmemPerCta ? 3
                                                                                   : 2;
}

template <int SRC, int NT, int XW>
struct Smem : SmemAt<SRC, NT, XW, ring_stages<SRC, NT, XW>()> {
  static constexpr int kStages = ring_stages<SRC, NT, XW>();
  static_assert(SmemAt<SRC, NT, XW, 2>::kBytes <= kSmemPerCta, "two stages must fit");
};

template <int SRC, int NT, int XW>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    gemv_kernel(const __grid_constant__ GemvBatch p, const __grid_constant__ TmaBatch tm, uint32_t total_units, int B,
                uint32_t* __restrict__ slot, uint32_t* __restrict__ err, const __grid_constant__ XtBatch xt) {
  static_assert(XW == 0 || SRC == kK15, "the transposed-x corrections are K15's");
  using S = Smem<SRC, NT, XW>;
  constexpr int kStages = S::kStages;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // the dynamic base is only guaranteed 16-byte aligned: round it up
  const uint32_t base_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((base_u32 + 1023) & ~1023u) - base_u32;
  uint8_t* smem = smem_raw + pad;
  // Two sets of partial tiles and corrections, alternating by unit parity, so
  // one barrier per unit suffices: a set is rewritten two units later, after
  // every thread has passed the next unit's barrier and so finished reading it.
  float* part = reinterpret_cast<float*>(smem + S::kPartOff);  // [2][warp][lane][4 NT]
  float* corr = reinterpret_cast<float*>(smem + S::kCorrOff);  // [2][...]
  uint32_t& first_unit = *reinterpret_cast<uint32_t*>(smem + S::kUnitOff);
  uint32_t* next_unit = reinterpret_cast<uint32_t*>(smem + S::kUnitOff + 4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ring = base_u32 + pad + uint32_t(warp) * kStages * StageGeom<SRC>::kBytes;
  const uint32_t bars = base_u32 + pad + S::kBarOff + uint32_t(warp) * kStages * 8;
  if (lane == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init_u32(bars + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // K15 with the transposed x (B = 3..8) and the plain GEMV at B = 9..16: the
  // warps of unit u walk their k-ranges from offset 7u (mod the range), so
  // that the CTAs do not all read the same lines of x at the same moment
  // (16384 x 53248: K15 B = 4 364 -> 331 us, B = 8 397 -> 385 us; plain B = 9
  // 305 -> 286 us, B = 16 356 -> 347 us).  The offset depends on the unit
  // only, so the order of every sum, and the result, is the same on every
  // call.  Elsewhere the walk made no gain or lost: the L1 prefetch of x at
  // B <= 8 already hides those reads (byte-split B = 1 216 -> 223 us with it),
  // K15 at B = 9..16 lost 6 %, and byte-split at B = 9..16 gained 1-3 % on
  // that weight but lost 2 % on a layer's matrices.
  constexpr bool kRot = (SRC == kK15 && (XW == 4 || XW == 8)) || (SRC == kPlain && NT == 2);
  constexpr uint32_t rot_mul = kRot ? 7u : 0u;
  // Every CTA starts on its own unit; the rest come from the counter, so a
  // launch with fewer than two units per CTA never leaves one CTA holding two
  // units while another has none.  A launch with a CTA for every unit leaves
  // the counter alone (no round trips to it; it stays zero).
  const bool counted = gridDim.x < total_units;
  auto grab = [&]() -> uint32_t { return counted ? gridDim.x + atomicAdd(slot, 1u) : total_units; };
  if (threadIdx.x == 0) {
    first_unit = blockIdx.x;
    next_unit[1] = grab();
  }
  __syncthreads();
  uint32_t* lut_w = reinterpret_cast<uint32_t*>(smem + S::kLutOff);
  constexpr int kRep = lut_rep<SRC, NT, XW>();
  const uint32_t lut = base_u32 + pad + S::kLutOff + uint32_t(lane % (kRep ? kRep : 1)) * 4;
  // the code-pair table of tensor ti, every thread writing its share
  auto build_lut = [&](int ti) {
    if constexpr (kRep > 0) {
      const RegTable& t = p.d[ti].t;
      for (uint32_t i = threadIdx.x; i < 256u * kRep; i += kThreads) {
        const uint32_t v = i / kRep, c0 = v & 15, c1 = v >> 4;
        const uint32_t h0 = (t.hi[c0 >> 2] >> (8 * (c0 & 3))) & 0xFF, e0 = (t.e0[c0 >> 2] >> (8 * (c0 & 3))) & 0x80;
        const uint32_t h1 = (t.hi[c1 >> 2] >> (8 * (c1 & 3))) & 0xFF, e1 = (t.e0[c1 >> 2] >> (8 * (c1 & 3))) & 0x80;
        lut_w[i] = e0 | (h0 << 8) | (e1 << 16) | (h1 << 24);
      }
    }
  };
  if (first_unit < total_units) {
    build_lut(owner(p.set_prefix, p.count, first_unit));
    __syncthreads();
  }
  // This thread's share of the escape corrections: row cj = tid / 16 of the
  // unit, batch slot cb, part cq of cP (cbp batch slots, cP = 16 / cbp parts),
  // so the 16 threads of a row read consecutive escapes of it.
  const int cbp = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
  const int cP = kThreads / (kRows * cbp);
  const int cj = threadIdx.x >> 4, cb = (threadIdx.x & 15) / cP, cq = (threadIdx.x & 15) % cP;
  uint32_t u = first_unit, u_next = next_unit[1];
  uint32_t issued = 0, done = 0;  // k-blocks copied / computed by this warp
  bool aborted = false;           // a wait ran out (warp-uniform): no more copies or waits, finish the schedule
#if WCOMP_DEBUG
  const bool skip_first_copy = g_debug_skip_first_copy != 0;
#else
  constexpr bool skip_first_copy = false;
#endif
  if (u < total_units) {
    Unit cur, nxt;
    uint32_t ce0 = 0, ce1 = 0, ne0 = 0, ne1 = 0;  // row cj's escapes in the current / next unit
    auto row_escapes = [&](const Unit& m, uint32_t& e0, uint32_t& e1) {
      if (SRC == kPlain || cj >= m.rows) {
        e0 = e1 = 0;
        return;
      }
      const TensorDesc& d = p.d[m.ti];
      e0 = d.row_index[m.r0 + cj];
      e1 = d.row_index[m.r0 + cj + 1];
    };
    unit_of(p, u, 0, warp, cur, rot_mul);
    row_escapes(cur, ce0, ce1);
    bool have_next = u_next < total_units;
    if (have_next) {
      unit_of(p, u_next, cur.ti, warp, nxt, rot_mul);
      row_escapes(nxt, ne0, ne1);
    }
    // The copy cursor: the next k-block to copy, in `cur` (ahead == 0) or
    // `nxt` (ahead == 1); it stops at the end of `nxt`.  Item i (the i-th
    // k-block this warp copies) uses stage i % kStages, whose mbarrier then
    // completes its phase i / kStages.
    int ahead = 0;
    uint32_t ckb = cur.kb0;
    auto issue_next = [&]() -> bool {
      if (ahead == 0 && ckb >= cur.kb1) {
        if (!have_next) return false;
        ahead = 1;
        ckb = nxt.kb0;
      }
      if (ahead == 1 && ckb >= nxt.kb1) return false;
      if (lane == 0 && !(skip_first_copy && issued == 0)) {
        const uint32_t sidx = issued % kStages;
        issue_item<SRC>(tm, ahead == 0 ? cur : nxt, kRot ? kb_at(ahead == 0 ? cur : nxt, ckb) : ckb, ring + sidx * StageGeom<SRC>::kBytes, bars + 8 * sidx);
      }
      ++issued;
      ++ckb;
      return true;
    };
    // Ask L2 for a unit's escape positions and values (two bulk prefetches),
    // so that the corrections find them there: a unit ahead where the whole
    // grid streams less than the L2 holds in one unit (span: every CTA's rows
    // times K at 1.5 bytes an element), at the unit's start where it streams
    // less than twice that (the corrections use a unit's escapes in the first
    // half of its k-loop), and not at all past that, where the prefetched
    // lines are evicted before use and read twice (16384 x 53248, K15, B = 1:
    // 305 -> 297 us without the prefetch; 6144 x 16384, B = 16: 91.6 -> 87.5
    // us with it).  `late`: the unit is starting and was not prefetched ahead.
    auto prefetch_escapes = [&](const Unit& m, bool ahead, bool late) {
      if (SRC == kPlain || threadIdx.x != 0) return;
      const TensorDesc& dm = p.d[m.ti];
      const uint64_t span = uint64_t(gridDim.x) * kRows * uint64_t(dm.K) * 3 / 2;
      if (ahead ? span > p.l2_bytes : (span > 2 * p.l2_bytes || (late && span <= p.l2_bytes))) return;
      const uint64_t e0 = dm.row_index[m.r0], e1 = dm.row_index[m.r0 + m.rows];
      if (e0 == e1) return;
      // the ranges end inside the padded position and value sections
      if (!WCOMP_DCHECK(e0 < e1 && e1 <= dm.E, 1)) return;
      const uint32_t vb = 2;  // bytes per escape value
      const uint64_t plo = (4 * e0) & ~uint64_t(15), phi = (4 * e1 + 15) & ~uint64_t(15);
      const uint64_t vlo = (vb * e0) & ~uint64_t(15), vhi = (vb * e1 + 15) & ~uint64_t(15);
      prefetch_l2(reinterpret_cast<const uint8_t*>(dm.esc_pos) + plo, uint32_t(phi - plo));
      prefetch_l2(reinterpret_cast<const uint8_t*>(dm.esc_val) + vlo, uint32_t(vhi - vlo));
    };
    prefetch_escapes(cur, false, false);
    if (have_next) prefetch_escapes(nxt, true, false);
    int par = 0;
    uint32_t grabbed = 0;
    if (threadIdx.x == 0) grabbed = grab();
    while (true) {
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      const TensorDesc& d = p.d[cur.ti];
      // ---- escape corrections of this unit, run through the k-loop.  Thread
      // (row cj, batch slot cb, part cq) owns the entries e = ce0 + cq + j cP
      // of row cj; with the transposed x, thread (cj, part tid % 16) owns
      // e = ce0 + part + 16 j and adds each to every batch row at once.  K15
      // up to 8 batch rows moves aligned quads instead: the part's quads start
      // at (ce0 rounded down to 4) + 4 (part + j parts).  Each k-block moves
      // esc_q entries one stage along: A requests the positions and values, B
      // (one k-block later) gathers x, C (one more k-block later) accumulates,
      // so every load has a k-block's compute to land.  What the loop does
      // not reach is taken after it.
      constexpr bool kXt = XW > 0;
      constexpr bool kQuads = SRC == kK15 && XW <= 8;  // K15 entries in aligned quads
      constexpr int kQ = esc_q<SRC, NT, XW>();
      constexpr int kXWords = kXt ? XW / 2 : 1;
      const uint64_t rowbase = uint64_t(cur.r0 + cj) * uint64_t(d.K);
      const uint32_t e_step = kXt ? uint32_t(kThreads / 16) : uint32_t(cP);
      uint32_t e_next = kXt ? ce0 + (threadIdx.x & 15) : ce0 + cq;
      const uint32_t e_end = SRC != kPlain && cj < cur.rows && (kXt || cb < B) ? ce1 : 0;
      const uint16_t* xrow = kXt ? xt.p[cur.ti] : p.x[cur.ti] + int64_t(cb) * d.K;
      uint32_t posA[kQ], valA[kQ], okA = 0, okB = 0;  // stage masks: entries requested / gathered
      uint32_t xB[kQ][kXWords], valB[kQ];
      float c = 0.f, cs[kXt ? XW : 1];
      // the quads: stage A's request, stage B's gathered x and values
      // (entries outside the row zeroed)
      uint32_t q_next = (ce0 & ~3u) + 4u * uint32_t(kXt ? (threadIdx.x & 15) : cq), qA = 0;
      const uint32_t q_step = 4u * uint32_t(kXt ? 16 : cP);
      uint4 pA = make_uint4(0u, 0u, 0u, 0u);
      uint2 vA = make_uint2(0u, 0u), vB = make_uint2(0u, 0u);
      uint32_t xQ[4][kXWords];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int w = 0; w < kXWords; ++w) xQ[i][w] = 0u;
      // Quad q's positions and values: aligned vector loads (a quad that
      // starts below E ends inside the position and value sections, which are
      // padded to 32 bytes).
      auto quad_load = [&](uint32_t q, uint4& pq, uint2& vq) {
        if (!WCOMP_DCHECK(q < d.E, 1)) q = 0;
        pq = *reinterpret_cast<const uint4*>(d.esc_pos + q);
        vq = *reinterpret_cast<const uint2*>(d.esc_val + q);
      };
      // Gather x for the quad's entries; entries outside [ce0, ce1) (only in
      // the row's first and last quads) read column 0 and get value 0 and x 0.
      auto quad_gather = [&](uint32_t q, const uint4& pq, uint2 vq, uint32_t (&xq)[4][kXWords], uint2& vout) {
        const uint32_t rb = uint32_t(rowbase);
        uint32_t k[4] = {pq.x - rb, pq.y - rb, pq.z - rb, pq.w - rb};
        uint32_t live = 0xFu;
        if (q < ce0 || q + 4u > ce1) {
          const uint32_t lo = q < ce0 ? ce0 - q : 0u, hi = q + 4u > ce1 ? ce1 - q : 4u;
          live = (0xFu << lo) & (0xFu >> (4u - hi));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (!((live >> i) & 1u)) k[i] = 0u;
          vq.x &= ((live & 1u) ? 0xFFFFu : 0u) | ((live & 2u) ? 0xFFFF0000u : 0u);
          vq.y &= ((live & 4u) ? 0xFFFFu : 0u) | ((live & 8u) ? 0xFFFF0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (!WCOMP_DCHECK(uint64_t(k[i]) < uint64_t(d.K), 1)) k[i] = 0u;
          if constexpr (XW == 0) {
            xq[i][0] = xrow[k[i]];
          } else if constexpr (XW == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(xrow + uint64_t(k[i]) * XW);
            xq[i][0] = v.x;
            xq[i][1 % kXWords] = v.y;
          } else {
            const uint4 v = *reinterpret_cast<const uint4*>(xrow + uint64_t(k[i]) * XW);
            xq[i][0] = v.x;
            xq[i][1 % kXWords] = v.y;
            xq[i][2 % kXWords] = v.z;
            xq[i][3 % kXWords] = v.w;
          }
        }
        if (live != 0xFu) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int w = 0; w < kXWords; ++w)
              if (!((live >> i) & 1u)) xq[i][w] = 0u;
        }
        vout = vq;
      };
      auto quad_accumulate = [&](const uint32_t (&xq)[4][kXWords], uint2 vq) {
        float dl[4];
        esc_delta_pair<SRC>(vq.x, dl[0], dl[1]);
        esc_delta_pair<SRC>(vq.y, dl[2], dl[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (kXt) {
#pragma unroll
            for (int h = 0; h < kXWords; ++h) {
              cs[2 * h] = fmaf(bf16_lo(xq[i][h]), dl[i], cs[2 * h]);
              cs[2 * h + 1] = fmaf(bf16_hi(xq[i][h]), dl[i], cs[2 * h + 1]);
            }
          } else {
            c = fmaf(__uint_as_float(xq[i][0] << 16), dl[i], c);
          }
        }
      };
#pragma unroll
      for (int b = 0; b < (kXt ? XW : 1); ++b) cs[b] = 0.f;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        posA[q] = uint32_t(rowbase);
        valA[q] = valB[q] = 0u;
#pragma unroll
        for (int w = 0; w < kXWords; ++w) xB[q][w] = 0u;
      }
      // stage A: request positions and values of the next kQ escapes
      auto esc_request = [&]() {
        if constexpr (kQuads) {
          okA = 1;
          qA = q_next;
          quad_load(q_next, pA, vA);
          q_next += q_step;
        } else if constexpr (SRC != kPlain) {
          okA = 0;
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const uint32_t i = e_next + q * e_step;
            const bool ok = i < e_end && WCOMP_DCHECK(i < d.E, 1);
            okA |= uint32_t(ok) << q;
            posA[q] = ok ? d.esc_pos[i] : uint32_t(rowbase);
            valA[q] = ok ? load_esc_val(d, i) : 0u;  // value 0 and x 0: contributes exactly 0
          }
          e_next += kQ * e_step;
        }
      };
      // stage C then B: accumulate the gathered escapes, gather the requested ones
      auto esc_advance = [&]() {
        if constexpr (kQuads) {
          if (okB) quad_accumulate(xQ, vB);
          if (okA) quad_gather(qA, pA, vA, xQ, vB);
          okB = okA;
          okA = 0;
        } else if constexpr (SRC != kPlain) {
          if (!(okA | okB)) return;  // nothing in flight (most k-blocks for byte-split's rare escapes)
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            if constexpr (kXt) {
              const float delta = esc_delta<WCOMP_K15>(valB[q]);
#pragma unroll
              for (int h = 0; h < kXWords; ++h) {
                cs[2 * h] = fmaf(bf16_lo(xB[q][h]), delta, cs[2 * h]);
                cs[2 * h + 1] = fmaf(bf16_hi(xB[q][h]), delta, cs[2 * h + 1]);
              }
            } else {
              c = fmaf(__uint_as_float(xB[q][0] << 16), esc_delta<SRC>(valB[q]), c);
            }
          }
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const uint64_t k = uint64_t(posA[q]) - rowbase;
            const bool ok = ((okA >> q) & 1) && WCOMP_DCHECK(k < uint64_t(d.K), 1);
            valB[q] = ok ? valA[q] : 0u;
            if constexpr (kXt) {
              const uint16_t* xr = xrow + k * XW;
              if (XW == 4) {
                const uint2 v = ok ? *reinterpret_cast<const uint2*>(xr) : make_uint2(0u, 0u);
                xB[q][0] = v.x;
                xB[q][1 % kXWords] = v.y;
              } else if (XW == 16) {
                uint32_t r[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if (ok) ld_x_v8(xr, r);
#pragma unroll
                for (int h = 0; h < 8; ++h) xB[q][h % kXWords] = r[h];
              } else {
#pragma unroll
                for (int h = 0; h < XW / 8; ++h) {
                  const uint4 v = ok ? reinterpret_cast<const uint4*>(xr)[h] : make_uint4(0u, 0u, 0u, 0u);
                  xB[q][(4 * h) % kXWords] = v.x; xB[q][(4 * h + 1) % kXWords] = v.y;
                  xB[q][(4 * h + 2) % kXWords] = v.z; xB[q][(4 * h + 3) % kXWords] = v.w;
                }
              }
            } else {
              xB[q][0] = ok ? uint32_t(xrow[k]) : 0u;
            }
          }
          okB = okA;
          okA = 0;
        }
      };
      if (SRC != kPlain && (kQuads ? q_next : e_next) < e_end) esc_request();
      for (uint32_t kb = cur.kb0; kb < cur.kb1; ++kb) {
        // every lane is done with the stage of the previous k-block, which the
        // copies below may refill
        __syncwarp();
        while (!aborted && issued < done + kStages && issue_next()) {
        }
        uint4 xv[NT][4];
        const uint32_t kr = kRot ? kb_at(cur, kb) : kb;  // the k-block this step computes
        load_x<NT, NT == 1 && XW == 0>(p, cur, kr, B, lane, xv);
        const uint32_t sidx = done % kStages;
        if (!aborted && __any_sync(0xffffffffu, !mbar_wait_bounded(bars + 8 * sidx, (done / kStages) & 1))) {
          aborted = true;  // the warp stops copying and waiting, and still runs the same instructions
          if (lane == 0) atomicOr(err, 1u);
        }
        const uint32_t st = ring + sidx * StageGeom<SRC>::kBytes;
        if (kr + 1 < cur.nkb || cur.kvalid == kKBlock)
          compute_item<SRC, NT, true, kRep>(d.t, lut, st, lane, true, xv, acc);
        else
          compute_item<SRC, NT, false, kRep>(d.t, lut, st, lane, uint32_t(32 * (lane & 3)) < cur.kvalid, xv, acc);
        ++done;
        if constexpr (SRC != kPlain) {
          esc_advance();
          // no new requests in the last k-block: what is left goes to the batches below
          if (kb + 1 < cur.kb1 && (kQuads ? q_next : e_next) < e_end) esc_request();
        }
      }
      // ---- unit end: partial tiles, escape corrections, fixed-order sums
      float* pp = part + ((par * kWarps + warp) * 32 + lane) * 4 * NT;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) pp[4 * nt + r] = acc[nt][r];
      if constexpr (SRC != kPlain) {
        // what the loop has in flight (a request made before a k-loop of no
        // k-blocks too), then the escapes it did not reach
        esc_advance();
        esc_advance();
        if constexpr (XW > 0) {
          // thread (row cj, part tid % 16 of 16): every batch row at once
          // from the transposed x; the 16 parts of a row (one half-warp) are
          // summed by a fixed shuffle tree
          if constexpr (kQuads) {
            for (uint32_t q = q_next; q < e_end; q += q_step) {
              uint4 p0;
              uint2 v0, w0;
              uint32_t x0[4][kXWords];
              quad_load(q, p0, v0);
              quad_gather(q, p0, v0, x0, w0);
              quad_accumulate(x0, w0);
            }
          } else {
            constexpr int D = XW >= 16 ? kEscDepth / 4 : kEscDepth / 2;
            for (uint32_t e = e_next; e < e_end; e += D * e_step) {
              uint32_t pos[D], val[D];
#pragma unroll
              for (int v = 0; v < D; ++v) {
                const uint32_t i = e + v * e_step;
                bool ok = i < e_end && WCOMP_DCHECK(i < d.E, 1);
                pos[v] = ok ? d.esc_pos[i] : uint32_t(rowbase);
                ok = ok && WCOMP_DCHECK(uint64_t(pos[v]) - rowbase < uint64_t(d.K), 1);
                if (!ok) pos[v] = uint32_t(rowbase);
                val[v] = ok ? load_esc_val(d, i) : 0u;  // value 0: delta 0
              }
              uint32_t wv[D][XW / 2];
#pragma unroll
              for (int v = 0; v < D; ++v) {
                const uint16_t* xr = xrow + uint64_t(uint64_t(pos[v]) - rowbase) * XW;
                if (XW == 4) {
                  const uint2 q2 = *reinterpret_cast<const uint2*>(xr);
                  wv[v][0] = q2.x;
                  wv[v][1 % (XW / 2)] = q2.y;
                } else if (XW == 16) {
                  uint32_t r[8];
                  ld_x_v8(xr, r);
#pragma unroll
                  for (int h = 0; h < 8; ++h) wv[v][h % (XW / 2)] = r[h];
                } else {
#pragma unroll
                  for (int q = 0; q < XW / 8; ++q) {
                    const uint4 q4 = reinterpret_cast<const uint4*>(xr)[q];
                    wv[v][(4 * q) % (XW / 2)] = q4.x; wv[v][(4 * q + 1) % (XW / 2)] = q4.y;
                    wv[v][(4 * q + 2) % (XW / 2)] = q4.z; wv[v][(4 * q + 3) % (XW / 2)] = q4.w;
                  }
                }
              }
#pragma unroll
              for (int v = 0; v < D; ++v) {
                const float delta = esc_delta<WCOMP_K15>(val[v]);
#pragma unroll
                for (int h = 0; h < XW / 2; ++h) {
                  cs[2 * h] = fmaf(bf16_lo(wv[v][h]), delta, cs[2 * h]);
                  cs[2 * h + 1] = fmaf(bf16_hi(wv[v][h]), delta, cs[2 * h + 1]);
                }
              }
            }
          }
#pragma unroll
          for (int b = 0; b < (kXt ? XW : 1); ++b) {
#pragma unroll
            for (int o = 8; o; o >>= 1) cs[b] += __shfl_xor_sync(0xffffffffu, cs[b], o);
          }
          if ((lane & 15) == 0) {
#pragma unroll
            for (int b = 0; b < (kXt ? XW : 1); ++b) corr[(par * kRows + cj) * 16 + b] = cs[b];
          }
        } else {
          if constexpr (kQuads) {
            // two quads at a time, all their loads in flight together
            for (uint32_t q = q_next; q < e_end; q += 2u * q_step) {
              const bool two = q + q_step < e_end;
              uint4 p0, p1 = make_uint4(0u, 0u, 0u, 0u);
              uint2 v0, v1 = make_uint2(0u, 0u), w0, w1 = make_uint2(0u, 0u);
              uint32_t x0[4][kXWords], x1[4][kXWords] = {};
              quad_load(q, p0, v0);
              if (two) quad_load(q + q_step, p1, v1);
              quad_gather(q, p0, v0, x0, w0);
              if (two) quad_gather(q + q_step, p1, v1, x1, w1);
              quad_accumulate(x0, w0);
              if (two) quad_accumulate(x1, w1);
            }
          } else {
            // kEscDepth escapes at a time, all their loads in flight together
            // (positions and values, then the x gathers); entries past the row's
            // last escape contribute exactly zero
            for (uint32_t e = e_next; e < e_end; e += kEscDepth * e_step) {
              uint32_t pos[kEscDepth], val[kEscDepth], xw[kEscDepth], okm = 0;
  #pragma unroll
              for (int v = 0; v < kEscDepth; ++v) {
                const uint32_t i = e + v * e_step;
                bool ok = i < e_end && WCOMP_DCHECK(i < d.E, 1);
                pos[v] = ok ? d.esc_pos[i] : uint32_t(rowbase);
                ok = ok && WCOMP_DCHECK(uint64_t(pos[v]) - rowbase < uint64_t(d.K), 1);
                okm |= uint32_t(ok) << v;
                val[v] = ok ? load_esc_val(d, i) : 0u;
              }
  #pragma unroll
              for (int v = 0; v < kEscDepth; ++v) {
                const bool ok = (okm >> v) & 1;
                xw[v] = ok ? uint32_t(xrow[int64_t(uint64_t(pos[v]) - rowbase)]) : 0u;
              }
  #pragma unroll
              for (int v = 0; v < kEscDepth; ++v)
                c = fmaf(__uint_as_float(xw[v] << 16), esc_delta<SRC>(val[v]), c);
            }
          }
          corr[par * kThreads + threadIdx.x] = c;
        }
      }
      // the unit after next (requested when this unit started), published
      // with this unit's partial sums
      if (threadIdx.x == 0) next_unit[par] = grabbed;
      __syncthreads();
      if (threadIdx.x < kRows * B && int(threadIdx.x & 15) < cur.rows) {
        const int j = threadIdx.x & 15, b = threadIdx.x >> 4;
        const int nt = b >> 3, bb = b & 7;
        const int src_lane = (j & 7) * 4 + (bb >> 1), reg = 4 * nt + (j >> 3) * 2 + (bb & 1);
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) y += part[((par * kWarps + w) * 32 + src_lane) * 4 * NT + reg];
        if constexpr (SRC != kPlain) {
          if (XW > 0) {
            y += corr[(par * kRows + j) * 16 + b];
          } else {
            for (int q = 0; q < cP; ++q) y += corr[par * kThreads + j * 16 + b * cP + q];
          }
        }
        if (WCOMP_DCHECK(b < B && cur.r0 + j < d.N, 2)) p.y[cur.ti][int64_t(b) * d.N + cur.r0 + j] = y;
      }
      if (!have_next) break;
      // advance: the next unit becomes current, the copy cursor keeps its place.
      // Every thread is past this unit's barrier, so none still reads the
      // table; a new tensor gets its own before any warp decodes it.
      if (kRep && nxt.ti != cur.ti) {
        build_lut(nxt.ti);
        __syncthreads();
      }
      cur = nxt;
      ce0 = ne0;
      ce1 = ne1;
      if (ahead == 1) {
        ahead = 0;
      } else {
        ckb = cur.kb0;
      }
      u_next = next_unit[par];
      par ^= 1;
      if (threadIdx.x == 0) grabbed = grab();
      have_next = u_next < total_units;
      if (have_next) {
        unit_of(p, u_next, cur.ti, warp, nxt, rot_mul);
        row_escapes(nxt, ne0, ne1);
        prefetch_escapes(nxt, true, false);
      }
      prefetch_escapes(cur, false, true);
    }
  }
  // A warp that gave up waiting lets its copies in flight land (bounded)
  // before the CTA exits; otherwise every copy it issued has been waited for.
  if (aborted && lane == 0) {
    const uint64_t deadline = global_ns() + kWaitNs;
    for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
      mbar_wait_until(bars + 8 * (i % kStages), (i / kStages) & 1, deadline);
  }
  __syncwarp();
  // The last CTA to finish returns the counter slot to zero for the next launch.
  if (counted && threadIdx.x == 0) {
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
  const float delta = d.scheme == WCOMP_BYTESPLIT ? esc_delta<WCOMP_BYTESPLIT>(val) : esc_delta<WCOMP_K15>(val);
  const int64_t k = int64_t(uint64_t(p) - rowbase);
#pragma unroll
  for (int b = 0; b < BT; ++b)
    if (b < B) s[b] = fmaf(__uint_as_float(uint32_t(x[int64_t(b) * d.K + k]) << 16), delta, s[b]);
}

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

// Per-device scratch: kSlots work-counter pairs, zeroed once at allocation;
// each launch takes the next slot and its last CTA zeroes the slot again.
// The word after the slots is the device error word.
std::mutex g_scratch_mu;
uint32_t* g_scratch[64] = {nullptr};
std::atomic<uint32_t> g_slot_rr{0};

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

// The driver's tensor-map encoder, reached through the runtime (no link
// against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A stream of N rows of row_bytes bytes as a 2-D byte array, read in boxes of
// 16 rows by box_bytes (128-byte swizzled when `swizzle`).  Reads past the
// last row or column arrive as zeros.
bool byte_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes, bool swizzle) {
  const EncodeTiledFn f = tensor_map_encoder();
  if (!f || row_bytes % 16 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, uint32_t(kRows)};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The container's tensor maps, made once (the container is immutable).
// Byte-split needs K % 32 == 0, K15 K % 128 == 0 (plane C rows of K / 8 bytes
// must be a multiple of 16 bytes long); other shapes take the element path.
bool container_maps(const wcomp_container* c) {
  wcomp_container* cc = const_cast<wcomp_container*>(c);
  std::call_once(cc->tmap_once, [cc] {
    const Layout& L = cc->L;
    const uint64_t N = uint64_t(L.N), K = uint64_t(L.K);
    const uint8_t* m = cc->d_main;
    bool ok;
    if (L.scheme == WCOMP_BYTESPLIT)
      ok = K % kGroup == 0 && byte_map(&cc->tmap[0], m + L.off_codes, K / 2, N, 64, false) &&
           byte_map(&cc->tmap[1], m + L.off_raw, K, N, 128, true);
    else
      ok = K % 128 == 0 && byte_map(&cc->tmap[0], m + L.off_codes, K / 2, N, 64, false) &&
           byte_map(&cc->tmap[1], m + L.off_a, K / 2, N, 64, false) &&
           byte_map(&cc->tmap[2], m + L.off_b, K / 4, N, 32, false) &&
           byte_map(&cc->tmap[3], m + L.off_c, K / 8, N, 16, false);
    cc->tmap_ok = ok ? 1 : 0;
  });
  return cc->tmap_ok == 1;
}

// Units (16-row sets) of every tensor of the batch, as a prefix.
uint32_t unit_prefix(GemvBatch& b, const int64_t* Ns) {
  uint32_t units = 0;
  for (int j = 0; j < b.count; ++j) {
    b.set_prefix[j] = units;
    units += uint32_t(cdiv(uint64_t(Ns[j]), kRows));
  }
  b.set_prefix[b.count] = units;
  return units;
}

// CTAs of a GEMV launch of `units` units when `resident` CTAs fit at once.
// Up to two units per resident CTA, one CTA per unit: the kernel then leaves
// the unit counter alone, and the hardware hands a finished CTA's slot to a
// waiting one on whichever SM frees first (measured: 6144 x 16384, 384 units
// on 304 slots, byte-split B = 1 49.7 -> 39.8 us, K15 66.5 -> 56.2 us; 6144 x
// 6144 22.3 -> 19.1 and 29.1 -> 25.1 us).  Above that, one CTA per slot,
// each taking further units from the counter with the next unit's copies
// started early (a CTA per unit took the 16384 x 53248 weight's 1,024 units
// from 214 to 222 us, byte-split B = 1).
uint32_t gemv_grid(uint32_t units, uint32_t resident) {
  if (units <= 2 * resident) return units > 0 ? units : 1;
  return resident;
}

// Resident CTAs per SM of one instantiation on device `dev`, with its
// shared-memory limit set (an attribute of the function in that device's
// context): done once per instantiation and device; racing first calls do
// the same idempotent work.
constexpr int kPrepDevices = 64;
template <int SRC, int NT, int XW>
int prepare_kernel(int dev) {
  auto kern = gemv_kernel<SRC, NT, XW>;
  constexpr uint32_t smem = Smem<SRC, NT, XW>::kBytes;
  static std::atomic<int> per_sm_cache[kPrepDevices];
  const bool cached = dev >= 0 && dev < kPrepDevices;
  int per_sm = cached ? per_sm_cache[dev].load(std::memory_order_acquire) : 0;
  if (!per_sm) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess) return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm <= 0)
      per_sm = 1;
    if (cached) per_sm_cache[dev].store(per_sm, std::memory_order_release);
  }
  return per_sm;
}

template <int SRC, int NT, int XW>
int launch(GemvBatch& b, const TmaBatch& tm, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  const uint32_t units = unit_prefix(b, Ns);
  uint32_t* base = nullptr;
  int st = scratch(dev, &base);
  if (st != WCOMP_OK) return st;
  uint32_t* slot = nullptr;
  if ((st = counter_slot(dev, &slot)) != WCOMP_OK) return st;
  const int per_sm = prepare_kernel<SRC, NT, XW>(dev);
  if (per_sm < 0) return map_cuda(cudaGetLastError());
  XtBatch xt;
  memset(&xt, 0, sizeof(xt));
  uint16_t* xt_mem = nullptr;
  if (XW > 0) {
    // x transposed into pool memory (freed in stream order after the GEMV)
    uint64_t cols = 0;
    for (int j = 0; j < b.count; ++j) {
      xt.kprefix[j] = uint32_t(cols);
      cols += uint64_t(b.d[j].K);
    }
    if (cols >= (uint64_t(1) << 32)) return WCOMP_EUNSUPPORTED;
    xt.kprefix[b.count] = uint32_t(cols);
    xt.count = b.count;
    cudaError_t e = pool_alloc(reinterpret_cast<void**>(&xt_mem), cols * (XW > 0 ? XW : 1) * sizeof(uint16_t), s);
    if (e != cudaSuccess) return map_cuda(e);
    for (int j = 0; j < b.count; ++j) xt.p[j] = xt_mem + uint64_t(xt.kprefix[j]) * (XW > 0 ? XW : 1);
    const uint32_t blocks = uint32_t(std::min<uint64_t>(cdiv(cols, 256), uint64_t(sms) * 8));
    constexpr int kXw = XW > 0 ? XW : 4;
    transpose_x_kernel<kXw><<<blocks, 256, 0, s>>>(b, xt, B);
    count_launches(1);
  }
  const uint32_t grid = gemv_grid(units, uint32_t(per_sm * sms));
  b.l2_bytes = l2_size(dev);
  gemv_kernel<SRC, NT, XW><<<grid, kThreads, Smem<SRC, NT, XW>::kBytes, s>>>(b, tm, units, B, slot,
                                                                                     base + 2 * kSlots, xt);
  count_launches(1);
  const cudaError_t e = cudaGetLastError();
  if (xt_mem) cudaFreeAsync(xt_mem, s);
  return map_cuda(e);
}

// K15 at B >= 3 corrects its escapes from a transposed copy of x, as wide as
// the batch rounds up to (4, 8 or 16 values per column), so one thread adds an
// escape to every batch row with one 8-, 16- or 32-byte load; byte-split's
// few escapes gain nothing from it.
template <int SRC>
int dispatch_vec(GemvBatch& b, const TmaBatch& tm, const int64_t* Ns, int B, int dev, int sms, cudaStream_t s) {
  if constexpr (SRC == kK15) {
    // from B = 3 the corrections read the transposed x; at B = 2 gathering x
    // directly is faster (16384 x 53248: 357 -> 330 us) and needs no pre-pass
    if (B >= 3) {
      if (B <= 4) return launch<SRC, 1, 4>(b, tm, Ns, B, dev, sms, s);
      if (B <= 8) return launch<SRC, 1, 8>(b, tm, Ns, B, dev, sms, s);
      return launch<SRC, 2, 16>(b, tm, Ns, B, dev, sms, s);
    }
  }
  return B <= 8 ? launch<SRC, 1, 0>(b, tm, Ns, B, dev, sms, s) : launch<SRC, 2, 0>(b, tm, Ns, B, dev, sms, s);
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
  const CUtensorMap* maps;  // its tensor maps (vector path)
  int kind;                 // Src for the vector path, 3 + Src for the element path
};

int run_items(Item* items, int count, int B, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = sm_count(dev);
  // longest rows first: the tail of the dynamic schedule is made of short units
  std::stable_sort(items, items + count, [](const Item& a, const Item& b) { return a.d.K > b.d.K; });
  std::vector<TmaBatch> tmb(1);  // 16 KB: kept off the stack
  TmaBatch& tm = tmb[0];
  for (int kind = 0; kind < 6; ++kind) {
    GemvBatch bt;
    memset(&bt, 0, sizeof(bt));
    int64_t Ns[kMaxBatch];
    auto flush = [&]() -> int {
      if (!bt.count) return WCOMP_OK;
      int st;
      switch (kind) {
        case 0: st = dispatch_vec<kBytesplit>(bt, tm, Ns, B, dev, sms, s); break;
        case 1: st = dispatch_vec<kK15>(bt, tm, Ns, B, dev, sms, s); break;
        case 2: st = dispatch_vec<kPlain>(bt, tm, Ns, B, dev, sms, s); break;
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
      if (items[i].maps) memcpy(tm.m[bt.count], items[i].maps, 4 * sizeof(CUtensorMap));
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
    const bool vec = aligned16(xs[i]) && container_maps(cs[i]);
    items[i].maps = vec ? cs[i]->tmap : nullptr;
    items[i].kind = (vec ? 0 : 3) + cs[i]->L.scheme;
  }
  return run_items(items.data(), count, B, s);
}

int gemv_plain(const uint16_t* const* ws, const int64_t* Ns, const int64_t* Ks, const uint16_t* const* xs, int B,
               float* const* ys, int count, cudaStream_t s) {
  if (B < 1 || B > 16) return WCOMP_EINVAL;
  std::vector<Item> items(count);
  std::vector<CUtensorMap> maps(size_t(count) * 4);
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
    // rows of 2K bytes, read in two 128-byte boxes per k-block
    const bool vec = Ks[i] % kGroup == 0 && aligned16(xs[i]) &&
                     byte_map(&maps[4 * size_t(i)], ws[i], 2 * uint64_t(Ks[i]), uint64_t(Ns[i]), 128, true);
    items[i].maps = vec ? &maps[4 * size_t(i)] : nullptr;
    items[i].kind = vec ? kPlain : 3 + kPlain;
  }
  return run_items(items.data(), count, B, s);
}

}  // namespace

WCOMP_DEBUG_TAKE(debug_take_gemv)
}  // namespace wc

using namespace wc;

namespace wc {
namespace {
uint32_t* noalloc_error_word(int dev);
}  // namespace
}  // namespace wc

extern "C" int wcomp_device_check(void* stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  uint32_t* base = nullptr;
  int st = scratch(dev, &base);
  if (st != WCOMP_OK) return st;
  uint32_t* words[2] = {base + 2 * kSlots, noalloc_error_word(dev)};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool failed = false;
  for (uint32_t* w : words) {
    if (!w) continue;
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, w, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return map_cuda(e);
    if (word) {
      failed = true;
      e = cudaMemsetAsync(w, 0, sizeof(uint32_t), s);
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return map_cuda(e);
    }
  }
  if (failed) return WCOMP_ETIMEOUT;
  const uint32_t dbg = debug_take_decode() | debug_take_encode() | debug_take_gemv();
  return dbg ? WCOMP_EBOUNDS : WCOMP_OK;
}

extern "C" int wcomp_debug_skip_first_copy(int on) {
#if WCOMP_DEBUG
  const uint32_t v = on ? 1u : 0u;
  const cudaError_t e = cudaMemcpyToSymbol(g_debug_skip_first_copy, &v, sizeof(v));
  if (e == cudaSuccess) {
    const cudaError_t e2 = cudaDeviceSynchronize();
    if (e2 != cudaSuccess) return map_cuda(e2);
  }
  return e == cudaSuccess ? WCOMP_OK : map_cuda(e);
#else
  (void)on;
  return WCOMP_EUNSUPPORTED;
#endif
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
// allocates with cudaMalloc on first use, and for K15 at B >= 3 a transposed
// copy of x from its memory pool.  Some callers cannot let a library allocate
// device memory: a serving loop that fixed its memory budget up front, or
// code that must not meet the implicit device synchronisation that a first
// cudaMalloc (or any cudaFree) can bring.  wcomp_gemv_noalloc runs the same
// kernel with its counters in the static device array below and corrects K15
// escapes from x directly.  The array is part of the library image, so every
// GPU that loads the library keeps it until the process exits.  Every call
// shares it.
// ---------------------------------------------------------------------------
namespace wc {
namespace {

constexpr int kNoAllocWords = 64;  // 256 bytes: [0] work counter, [1] completion counter, [2] error word
// A call may cover at most this many rows: the work counter runs past the
// unit count by a few grabs per CTA of the grid and must stay within 32 bits.
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

// Its error word (word 2 of the array), once the array's address is known.
uint32_t* noalloc_error_word(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  return g_noalloc_ptr[dev] ? g_noalloc_ptr[dev] + 2 : nullptr;
}

template <int SRC, int NT>
int launch_on(GemvBatch& b, const TmaBatch& tm, int64_t N, int B, int dev, int sms, uint32_t* slot, cudaStream_t s) {
  const uint32_t units = unit_prefix(b, &N);
  const int per_sm = prepare_kernel<SRC, NT, 0>(dev);
  if (per_sm < 0) return map_cuda(cudaGetLastError());
  XtBatch xt;
  memset(&xt, 0, sizeof(xt));
  const uint32_t grid = gemv_grid(units, uint32_t(per_sm * sms));
  b.l2_bytes = l2_size(dev);
  gemv_kernel<SRC, NT, 0><<<grid, kThreads, Smem<SRC, NT, 0>::kBytes, s>>>(b, tm, units, B, slot, slot + 2, xt);
  count_launches(1);
  return map_cuda(cudaGetLastError());
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
  const bool vec = aligned16(d_x) && container_maps(c);
  if (!vec) {
    // the element path uses no scratch at all
    return c->L.scheme == WCOMP_BYTESPLIT ? dispatch_generic<kBytesplit>(b, &N, B, sms, s)
                                          : dispatch_generic<kK15>(b, &N, B, sms, s);
  }
  // the tensor maps travel as a kernel parameter (16 KB, kept off the stack)
  std::unique_ptr<TmaBatch> tm(new (std::nothrow) TmaBatch);
  if (!tm) return WCOMP_ENOMEM;
  memcpy(tm->m[0], c->tmap, sizeof(c->tmap));
  if (c->L.scheme == WCOMP_BYTESPLIT)
    return B <= 8 ? launch_on<kBytesplit, 1>(b, *tm, N, B, dev, sms, scratch, s)
                  : launch_on<kBytesplit, 2>(b, *tm, N, B, dev, sms, scratch, s);
  return B <= 8 ? launch_on<kK15, 1>(b, *tm, N, B, dev, sms, scratch, s) : launch_on<kK15, 2>(b, *tm, N, B, dev, sms, scratch, s);
}
