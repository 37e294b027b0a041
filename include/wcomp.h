/*
 * wcomp.h - lossless BF16 weight coding (byte-split and K15) with a standalone
 * decode and a fused decode-GEMV, for NVIDIA GB300 (sm_103a).
 *
 * The method.  "Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%"
 * (forgeeks.dev), section "Cómo funciona la compresión": a BF16 weight is
 * 1 sign, 8 exponent and 7 mantissa bits; trained weights reuse a narrow set
 * of sign+exponent symbols.
 *   - byte-split: the high byte (sign + exponent bits 7..1) becomes a 4-bit
 *     code into a per-tensor 15-entry dictionary, code 15 meaning "escape";
 *     escaped high bytes are kept exactly in a (position, byte) stream and
 *     the low byte is stored unchanged (12.005 bits/weight on the pages'
 *     checkpoint, every tensor bit-exact);
 *   - K15: the 9-bit sign+exponent symbol becomes a 4-bit code into a
 *     15-entry table with the same escape rule; the 7-bit mantissa is stored
 *     unchanged (11.173 bits/weight with all overhead on the pages' checkpoint).
 * "Compresión de pesos LLM sin pérdida vs 8-bit GGUF" (wavect.io), section
 * "¿Qué significa “sin pérdida” para los pesos de un LLM?": lossless means the
 * round trip rebuilds every bit; a GPU may keep the weights encoded and rebuild
 * exact BF16 in registers for the matrix product.  Section "Qué queda por
 * demostrar" of the forgeeks page names the open step this library builds: a
 * GEMV that rebuilds the weights in registers and applies the sparse escape
 * correction in the same kernel.
 *
 * Conventions for every entry point below.
 *   - Weights and activations are BF16 bit patterns passed as 16-bit words;
 *     the codec never does float arithmetic on weights, so NaN, Inf, -0 and
 *     subnormals round-trip.
 *   - A weight tensor is W[N, K], row-major (y = x W^T).  n = N * K must be
 *     in [1, 2^32); otherwise WCOMP_EUNSUPPORTED.
 *   - Pointers named d_* are device pointers on the current CUDA device and
 *     are owned by the caller.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).  Calls are stream-ordered and
 *     asynchronous unless stated otherwise.
 *   - Every call returns a wcomp_status and never aborts; CUDA errors are
 *     WCOMP_ECUDA.  A failed call leaves its outputs unspecified and frees
 *     what it allocated.
 *   - Containers are opaque, owned by the library, and released with
 *     wcomp_free.  A container lives on the device that was current when it
 *     was made.  Container memory comes from a stream-ordered memory pool the
 *     library creates per device; freed blocks stay in that pool for reuse
 *     until the process exits.
 */
#ifndef WCOMP_H
#define WCOMP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WCOMP_VERSION 1

#if defined(__GNUC__)
#define WCOMP_API __attribute__((visibility("default")))
#else
#define WCOMP_API
#endif

typedef enum { WCOMP_BYTESPLIT = 0, WCOMP_K15 = 1 } wcomp_scheme;

typedef enum {
  WCOMP_OK = 0,
  WCOMP_EINVAL = -1,        /* bad argument (null pointer, size, scheme, B) */
  WCOMP_ENOMEM = -2,        /* device or host allocation failed */
  WCOMP_ECORRUPT = -3,      /* serialized container failed validation */
  WCOMP_ECUDA = -4,         /* a CUDA runtime call failed */
  WCOMP_EUNSUPPORTED = -5,  /* size outside the supported range */
  WCOMP_ETIMEOUT = -6,      /* a kernel's bounded wait on its own copies ran out */
  WCOMP_EINTERNAL = -7,     /* an internal consistency check failed; no result was returned */
  WCOMP_EBOUNDS = -8        /* a debug build's index check failed inside a kernel (the access was skipped) */
} wcomp_status;

typedef struct wcomp_container wcomp_container;

/* Description of a container (filled by wcomp_info). */
typedef struct {
  int32_t scheme;            /* wcomp_scheme */
  int32_t version;           /* container format version */
  int64_t N, K, n;           /* shape and element count */
  uint64_t n_escapes;        /* E: elements whose symbol is not in the table */
  uint32_t tile_elems;       /* granule of the tile escape index (8192) */
  uint32_t n_tiles;
  uint16_t table[15];        /* the 15 symbols, most frequent first */
  uint16_t pad_;
  uint64_t bytes_codes;      /* 4-bit code stream */
  uint64_t bytes_raw;        /* raw low bytes (byte-split) or mantissa planes (K15) */
  uint64_t bytes_index;      /* tile and row escape indexes */
  uint64_t bytes_escapes;    /* escape positions and values */
  uint64_t serialized_bytes; /* header + padded payload */
  double entropy_bpw;        /* 4 + raw bits + (E + 15) * symbol bits / n */
  double physical_bpw;       /* 8 * serialized_bytes / n */
  uint64_t serialized_compact_bytes; /* header + padded payload of the compact form */
  double physical_compact_bpw;       /* 8 * serialized_compact_bytes / n */
} wcomp_info_t;

/*
 * Encode one BF16 tensor.
 *   d_w     device, uint16[N*K] row-major BF16 bits (any alignment; 16-byte
 *           aligned input takes the vector path).
 *   scheme  WCOMP_BYTESPLIT or WCOMP_K15.
 *   out     receives a new container (NULL on failure).
 * Steps (all on the GPU): per-tensor symbol histogram (256 or 512 bins),
 * table of the 15 most frequent symbols (count descending, symbol ascending),
 * 4-bit packing of codes and raw bits, per-tile escape counts and their scan,
 * escape compaction in ascending position order, tile and row escape indexes.
 * Waits on `stream` twice: once for the escape count the histogram implies,
 * which sizes the escape stream (the pack and scan kernels keep running
 * meanwhile), and once for the tile scan, whose total must equal that count
 * (else WCOMP_EINTERNAL and no container).  The escape compaction and the row
 * index are still running on `stream` when the call returns.  Output is
 * deterministic and byte-identical to the CPU oracle.
 * Definition: forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi
 * un 25%", section "Cómo funciona la compresión": the sign+exponent symbol
 * (8 bits for byte-split, 9 for K15) gets a 4-bit code into the tensor's
 * table of 15 symbols, code 15 marks an escape kept exactly, the low byte or
 * 7-bit mantissa is stored as is.
 */
WCOMP_API int wcomp_encode(const uint16_t* d_w, int64_t N, int64_t K, int scheme, void* stream,
                 wcomp_container** out);

/*
 * How wcomp_encode_batched sizes its histogram grid (host-side, no device
 * work; exposed so the sizing can be checked without a GPU).  n[i] is the
 * element count of tensor i of a batch whose tensors are all histogrammed,
 * sms the device's SM count; blocks[i] receives the number of 256-thread
 * blocks tensor i gets.  Thread t of block b counts the 8-element chunks
 * b * 256 + t, b * 256 + t + 256 * blocks[i], ...; the counters are 16-bit
 * halves shared by 8 threads, so no thread may be given more than 1023
 * chunks (8 x 8 x 1023 = 65472 elements per half).  Returns WCOMP_EINVAL for
 * a null pointer, count or sms <= 0, or an n outside [1, 2^32).
 */
WCOMP_API int wcomp_encode_hist_grid(const uint64_t* n, int count, int sms, uint32_t* blocks);

/*
 * Encode `count` tensors in one pass: tensor i is W_i[N[i], K[i]] at d_w[i],
 * coded with schemes[i]; out[i] receives its container.  The same steps as
 * wcomp_encode run as batched launches over all tensors, with the same two
 * waits on `stream` for the whole batch (escape counts, then the scan check).
 * The batch's containers share two pool blocks (one for their code, raw and
 * index sections, one for their escape streams); each container is still
 * released on its own with wcomp_free, and a block returns to the pool with
 * the last container that uses it.  On failure every out[i] is NULL.
 * Definition: as wcomp_encode (forgeeks page, "Cómo funciona la compresión";
 * one table per tensor).
 */
WCOMP_API int wcomp_encode_batched(const uint16_t* const* d_w, const int64_t* N, const int64_t* K,
                                   const int* schemes, int count, void* stream, wcomp_container** out);

/*
 * Decode a container to exact BF16 bits.
 *   d_out   device, uint16[N*K]; the caller's buffer.
 * The code stream is expanded through the 15-entry table, joined with the raw
 * bits, and escaped elements are patched from the escape stream.
 * Definition: forgeeks page, "Cómo funciona la compresión" (byte-split
 * reconstruction of the high byte; K15 symbol + mantissa).
 */
WCOMP_API int wcomp_decode(const wcomp_container* c, uint16_t* d_out, void* stream);

/*
 * Fused decode-GEMV:  y[b, r] = sum_k x[b, k] * W[r, k]  for b < B, r < N.
 *   d_x     device, uint16[B*K] BF16 bits, row-major, contiguous.
 *   B       batch, 1 <= B <= 16.
 *   d_y     device, float[B*N], row-major; overwritten.
 * W is rebuilt in registers from the codes and raw bits; escaped weights are
 * corrected inside the same kernel (y += x * (w_true - w_placeholder)).
 * Products run on the tensor cores (BF16 MMAs with fp32 accumulation); the
 * summation order is fixed (no atomics), so repeated calls give identical
 * bits.  Shapes with K % 32 != 0 (K15: K % 128 != 0) or an x that is not
 * 16-byte aligned take a slower element-by-element path with the same result
 * contract.
 * Memory: the work counters live in a device buffer the library allocates
 * with cudaMalloc on first use per device; a K15 container at B >= 3 also
 * takes a transposed copy of x (K * 4..16 * 2 bytes) from the library's
 * stream-ordered pool for the duration of the call.  wcomp_gemv_noalloc
 * allocates nothing.
 * Errors found on the device (a copy that never completed) do not fail the
 * call: the kernel records them and stops waiting; wcomp_device_check
 * reports them.
 * Definition: forgeeks page, "Qué queda por demostrar" (GEMV on codes rebuilt
 * in registers, escape correction); wavect page on rebuilding exact BF16 in
 * registers for the matmul.
 */
WCOMP_API int wcomp_gemv(const wcomp_container* c, const uint16_t* d_x, int B, float* d_y, void* stream);

/*
 * wcomp_gemv without any allocation.  The method on the pages has no
 * counterpart to this entry point; it exists for callers that cannot let the
 * library allocate device memory: a serving loop that fixed its memory budget
 * up front, or code that must not meet the implicit device synchronisation a
 * first cudaMalloc or any cudaFree can bring.  wcomp_gemv takes its work
 * counters from a buffer it allocates on first use; this variant keeps them
 * in a 256-byte static device array inside the library instead, which every
 * GPU that loads the library holds until the process exits.
 *   Arguments and results are those of wcomp_gemv.
 *   The first call on a device looks up the array's device address (a
 *   host-side runtime query, no allocation); make that first call before any
 *   stream capture.
 *   Every call shares the one array and zeroes its counters in stream order
 *   before the kernel starts: calls whose kernels overlap on the GPU (on
 *   different streams) race and must be ordered by the caller.
 *   A call covers at most 2^31 - 2^20 rows (N); larger N returns
 *   WCOMP_EUNSUPPORTED.  No cudaMalloc, cudaFree or other allocating routine
 *   is called.
 */
WCOMP_API int wcomp_gemv_noalloc(const wcomp_container* c, const uint16_t* d_x, int B, float* d_y, void* stream);

/*
 * Plain BF16 GEMV over an uncompressed W[N, K] with the same contract as
 * wcomp_gemv; the comparison kernel for the fused path ("0.733x the BF16 GEMV
 * time", forgeeks page, "Qué queda por demostrar").
 */
WCOMP_API int wcomp_gemv_bf16(const uint16_t* d_w, int64_t N, int64_t K, const uint16_t* d_x, int B,
                    float* d_y, void* stream);

/*
 * Batched plain BF16 GEMV: tensor i is W_i[N[i], K[i]] at d_w[i] with input
 * d_x[i] (B x K[i]) and output d_y[i] (B x N[i]); host arrays of length count.
 * The same launch structure as wcomp_gemv_batched, so the two compare like
 * for like.
 */
WCOMP_API int wcomp_gemv_bf16_batched(const uint16_t* const* d_w, const int64_t* N, const int64_t* K,
                                      const uint16_t* const* d_x, int B, float* const* d_y, int count,
                                      void* stream);

/*
 * Batched forms: one launch over `count` containers (any mix of schemes and
 * shapes).  Arrays are host arrays of length count; every d_outs[i] /
 * d_x[i] / d_y[i] is a device buffer sized for containers[i].  All
 * containers must live on the current device.  count may be any positive
 * number (large batches are split into several launches).
 */
WCOMP_API int wcomp_decode_batched(const wcomp_container* const* containers, uint16_t* const* d_outs,
                         int count, void* stream);
WCOMP_API int wcomp_gemv_batched(const wcomp_container* const* containers, const uint16_t* const* d_x,
                       int B, float* const* d_y, int count, void* stream);

/*
 * Report and clear the device error words of the current device (the one
 * wcomp_gemv and the batched GEMVs use, and the one in wcomp_gemv_noalloc's
 * static array).  A GEMV kernel whose bounded wait on its own tensor copies
 * runs out records it there and finishes without waiting instead of hanging;
 * its outputs are then undefined.  In a debug build (compiled with
 * WCOMP_DEBUG=1) the kernels also check their indexes before memory
 * accesses, skip an access that fails and record it.  Synchronizes `stream`.
 * Returns WCOMP_OK, WCOMP_ETIMEOUT or WCOMP_EBOUNDS.
 */
WCOMP_API int wcomp_device_check(void* stream);

/*
 * Test hook for the bounded waits, in debug builds only (compiled with
 * WCOMP_DEBUG=1).  While `on` is non-zero, every warp of a GEMV launch
 * (fused or plain) leaves the first of its tensor copies unissued but still
 * waits for it: the wait runs out after about a second, the warp stops
 * copying and waiting, lets the copies it has in flight land and finishes,
 * and wcomp_device_check then reports WCOMP_ETIMEOUT.  The outputs of such a
 * launch are undefined; the context stays usable.  Applies to the current
 * device and synchronizes it.  Release builds do nothing and return
 * WCOMP_EUNSUPPORTED.  (Library housekeeping; the pages define no
 * counterpart.)
 */
WCOMP_API int wcomp_debug_skip_first_copy(int on);

/*
 * Describe a container (host-side, no device work): shape, table, section
 * sizes, and the bits/weight accounting of forgeeks page "Prueba de GLM-5.2
 * reduce la memoria BF16 en casi un 25%", section "Cómo funciona la
 * compresión" (a 4-bit code plus 8 raw bits for byte-split or 7 for K15 per
 * weight, plus each escape and each table entry at its symbol width), next to
 * the physical bits/weight of both serialized forms.  Returns WCOMP_EINVAL
 * for a NULL argument.
 */
WCOMP_API int wcomp_info(const wcomp_container* c, wcomp_info_t* info);

/*
 * Serialize to a host buffer: a 96-byte header (magic "WCMP", version,
 * scheme, N, K, E, tile size, table, payload length, CRC-32 of the payload,
 * CRC-32 of the header) followed by the payload sections, each padded to 32
 * bytes.  With host_buf == NULL only *len is set.  Returns WCOMP_EINVAL if
 * cap is too small.  Synchronizes `stream`.  The pages fix no file format;
 * this one stores every section the device container holds, so that
 * wcomp_deserialize rebuilds it without recomputation, and carries checksums
 * for the corruption checks of wavect page "Compresión de pesos LLM sin
 * pérdida vs 8-bit GGUF", section "Un piloto de producción de 14 días".
 */
WCOMP_API int wcomp_serialize(const wcomp_container* c, void* host_buf, uint64_t cap, uint64_t* len,
                    void* stream);

/*
 * Serialize to the compact form (format version 2): the same header, then
 * the code stream, the raw bytes (byte-split) or the three K15 mantissa
 * planes, one little-endian uint16 escape count per 8192-element tile, and
 * the escape symbols in ascending position order (byte-split: one byte, the
 * high byte; K15: the 9-bit sign+exponent symbol, packed least significant
 * bit first so that symbol r occupies stream bits 9r .. 9r+8).  Positions,
 * the row index and the K15 escape mantissas are implied (by the codes 15
 * and the planes), so the physical size tracks the bits/weight accounting of
 * forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%",
 * section "Cómo funciona la compresión", which counts each escape at its
 * symbol width.  Sections are padded to 32 bytes with zeros.  With host_buf
 * == NULL only *len is set.  Returns WCOMP_EINVAL if cap is too small.
 * Synchronizes `stream`.
 */
WCOMP_API int wcomp_serialize_compact(const wcomp_container* c, void* host_buf, uint64_t cap, uint64_t* len,
                                      void* stream);

/*
 * Rebuild a container from serialized bytes (host buffer), either form.
 * Version 1: the header, both checksums, the section sizes, the escape
 * positions (strictly ascending, below n), both escape indexes and the
 * agreement between escape codes and positions are validated on the host.
 * Version 2 (compact): the header, both checksums and the section sizes are
 * validated, the positions are rebuilt from the codes 15 and must number E,
 * and every tile's escape count must match.  Nothing is copied to the device
 * unless every check passes; any mismatch returns WCOMP_ECORRUPT ("inject
 * corruption" and "validate hashes", wavect page, "Un piloto de producción
 * de 14 días").  Both forms give the same device container.  Synchronizes
 * `stream`.
 */
WCOMP_API int wcomp_deserialize(const void* host_buf, uint64_t len, void* stream, wcomp_container** out);

/*
 * Release a container.  The device memory is returned in stream order on
 * `stream`: work queued earlier on that stream may still use it.  Containers
 * made by one wcomp_encode_batched call share their blocks, which return to
 * the pool on the stream of the last wcomp_free among them: a caller that
 * frees them on different streams orders those streams first.  NULL is a
 * no-op.  (Library housekeeping; the pages define no counterpart.)
 */
WCOMP_API void wcomp_free(wcomp_container* c, void* stream);

/* Human-readable text for a status code (static string). */
WCOMP_API const char* wcomp_strerror(int status);

/* WCOMP_VERSION of the library that was loaded. */
WCOMP_API int wcomp_version(void);

/*
 * Number of CUDA kernels this library has launched in the calling process
 * (all devices, all threads).  Host-side counter, no device work; used to
 * report how many of the library's own kernels a timed region ran.
 */
WCOMP_API uint64_t wcomp_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* WCOMP_H */
