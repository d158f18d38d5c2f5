/*
 * qps.h: C ABI of the position-split, quantised-KV decode-attention library.
 *
 * The library computes decode attention (one, or a few verify, query tokens per
 * sequence) over a KV cache that is split
 * by key position into a device-resident window [0, wc) and a host-resident tail
 * [wc, n_kv).  Each part runs a split-KV flash-decode that emits a normalised output
 * and its log-sum-exp (LSE); the parts are merged by an LSE combine.  K and V may be
 * stored compressed (K: q8_0; V: q8_0 or 3-bit TurboQuant-MSE) and are dequantised on
 * read inside the attention loop.  The tail streams from pinned host memory through a
 * ring of device staging slots filled on a copy stream.
 *
 * Sources (page title, section):
 *   [RKV]  "F5 M7 — Rolling KV: position-windowed KV residency": header status block
 *          (position split, LSE-emitting attention) and section "Implementation
 *          decomposition, refined (S1 -> S2 -> S3)", item S2 (per-tile O_t, lse_t and
 *          the f32 merge; a single tile is plain attention).
 *   [RING] "Rolling-KV: step/graph-level tail prefetch (design)", section "The fix: a
 *          persistent, step-spanning tail-prefetch ring" (B = 2..4 slots sized once,
 *          a flat (layer, tile) schedule kept B ahead on a copy stream, copy_done /
 *          compute_done events instead of a per-op barrier, pre-created events).
 *   [POLY] "F5 M6 — PolyKV (shared compressed KV pool)": section "What PolyKV is
 *          (reference)" (K int8 / V 3-bit TurboQuant-MSE), section "S1 — SharedKVPool"
 *          (one prefix read by many agents), section "S2 perf-path Level B" (V read as
 *          centroid x norm in the rotated domain, output inverse-rotated once), and
 *          section "S2 perf-path — turbo-MMA verify kernel + scalar-K/turbo-V fused
 *          decode" (n_q > 1 query tokens per sequence on tensor cores, K / V
 *          dequantised in the tile).
 *   [TSTAR] "T*-aware auto rolling-KV spill (HAL #582 P1+, #621 follow-on)": sections
 *          "The decision (fit-condition reformulation)" and "T* — the negligible-drop
 *          tail band" (per-token drop of a streamed tail, the largest tail T* within a
 *          target drop, the first storage tier that fits budget + T*).
 *
 * Conventions shared by every call:
 *   - Every call returns a qps_status; qps_last_error() gives a thread-local message
 *     for the last failing call on the calling thread.  No call aborts, throws across
 *     the ABI, or traps on the device.
 *   - Pointers are raw.  "device" pointers are CUDA device memory of the current
 *     device (the caller owns them, e.g. PyTorch tensors); "host" pointers are host
 *     memory read synchronously during the call; "pinned" pointers are page-locked
 *     host memory (cudaHostAlloc / cudaHostRegister / torch pin_memory).
 *   - `stream` arguments are cudaStream_t values passed as void*; NULL is the legacy
 *     default stream.  Calls taking a stream only enqueue work on it and return
 *     without waiting for the device, unless stated otherwise.
 *   - fp16 data is IEEE binary16, stored as 2-byte little-endian values.
 *   - A "row" is one stored vector of head_dim values: one (token, KV head) of a K or
 *     V cache.  Views address rows by strides in rows; each storage plane has its own
 *     bytes per row (below), so one row index addresses every plane of a format.
 *   - Unsupported shapes or formats return QPS_ERR_UNSUPPORTED; there is no fallback
 *     path of any kind.
 *
 * Storage formats (bytes per row for head_dim D):
 *   QPS_FMT_F16   data: D fp16 values (2D bytes).
 *   QPS_FMT_Q8_0  data: D int8 codes (D bytes); aux: D/32 fp16 scales (D/16 bytes).
 *                 Value = code * scale of its 32-value block.
 *   QPS_FMT_TQ3   data: 2-bit magnitude plane (D/4 bytes); aux: 1-bit sign plane
 *                 (D/8 bytes); aux2: one fp16 L2 norm (2 bytes).  Element i is at bits
 *                 2(i%4)..2(i%4)+1 of byte i/4 and bit i%8 of byte i/8.  Level index
 *                 k = sign ? 4 + mag : 3 - mag; value = (norm / D) * s .* (H c[k]),
 *                 H the Sylvester-Hadamard matrix, s the seeded sign diagonal, c the
 *                 8-level codebook returned by qps_tq_codebook(3, ...).
 *   QPS_FMT_TQ2   data: 2-bit fields (sign << 1) | mag (D/4 bytes), element i at bits
 *                 2(i%4)..2(i%4)+1 of byte i/4; aux: one fp16 norm (2 bytes).
 *                 k = sign ? 2 + mag : 1 - mag over the 4-level codebook; value as TQ3.
 *   QPS_FMT_TQ4   data: 4-bit fields (sign << 3) | mag (D/2 bytes), element i at bits
 *                 4(i%2)..4(i%2)+3 of byte i/2; aux: one fp16 norm (2 bytes).
 *                 k = sign ? 8 + mag : 7 - mag over the 16-level codebook; value as TQ3.
 *   TQ2 / TQ3 / TQ4 are the 2-, 3- and 4-bit rungs of one rotation + codebook scheme
 *   [POLY, "S2 — TurboQuant tier family"]: V formats, and K formats where V is in the
 *   same tier.
 */
#ifndef QPS_H
#define QPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QPS_ABI_VERSION 7

#if defined(__GNUC__)
#define QPS_API __attribute__((visibility("default")))
#else
#define QPS_API
#endif

typedef enum qps_status {
  QPS_OK = 0,
  QPS_ERR_INVALID_ARG = 1, /* a pointer, size, stride, alignment or range is invalid */
  QPS_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim, format pairing) */
  QPS_ERR_CUDA = 3,        /* a CUDA runtime call failed; the message names it */
  QPS_ERR_TIMEOUT = 4,     /* a bounded host wait ran out */
  QPS_ERR_STATE = 5,       /* call out of order (ring schedule, destroyed object) */
  QPS_ERR_INTERNAL = 6     /* a consistency check inside the library failed */
} qps_status;

typedef enum qps_kv_format {
  QPS_FMT_F16 = 0,
  QPS_FMT_Q8_0 = 1,
  QPS_FMT_TQ3 = 2,
  QPS_FMT_TQ2 = 3,
  QPS_FMT_TQ4 = 4
} qps_kv_format;

/* ABI version of the loaded library (QPS_ABI_VERSION it was built with).  Library
 * utility, no counterpart on the pages.  Never fails. */
QPS_API int32_t qps_abi_version(void);

/* Message of the last failing call on this thread ("" if none).  The pointer stays
 * valid until the next failing call on the same thread.  Library utility, no
 * counterpart on the pages.  Never fails. */
QPS_API const char* qps_last_error(void);

/* Constant name of a status code ("QPS_OK", ...; "QPS_UNKNOWN_STATUS" for any other
 * value).  Library utility, no counterpart on the pages.  Never fails. */
QPS_API const char* qps_status_name(int32_t status);

/* The fixed TQ3 codebook [POLY, "S2 — TurboQuant tier family"]: the 8-level Lloyd-Max
 * quantiser of N(0,1), each level rounded to the nearest fp16 value, levels exactly
 * symmetric, thresholds the exact midpoints of adjacent levels.  Host only; needs no
 * GPU.  levels: host, 8 floats (ascending); thresholds: host, 7 floats.  Either may be
 * NULL.  Errors: none. */
QPS_API qps_status qps_tq3_codebook(float* levels, float* thresholds);

/* The codebook of the `bits`-bit TurboQuant tier (2, 3 or 4), built like the TQ3 one
 * from the 2^bits-level Lloyd-Max quantiser of N(0,1) [POLY, "S2 — TurboQuant tier
 * family"].  levels: host, 2^bits floats (ascending); thresholds: host, 2^bits - 1
 * floats; either may be NULL.  Host only.  Errors: UNSUPPORTED (bits). */
QPS_API qps_status qps_tq_codebook(int32_t bits, float* levels, float* thresholds);

/* q8_0 encode [POLY, "What PolyKV is (reference)"; problem statement: 32-value blocks,
 * fp16 scale = absmax / 127, int8 codes].
 *   x       device, fp16 rows [rows][D] with row stride x_row_stride (elements,
 *           multiple of 8, >= D); 16-byte aligned.
 *   codes   device, int8 [rows][D] contiguous; 8-byte aligned.
 *   scales  device, fp16 [rows][D/32] contiguous; 2-byte aligned.
 * Per block: d16 = fp16(f32(absmax) / 127); code = clamp(round_half_away(f32(x) /
 * f32(d16)), -127, 127), all IEEE float32; a block with d16 == 0 stores zero codes.
 * D in {32, 64, 128, 256, 512}.  rows == 0 is a no-op.
 * Errors: INVALID_ARG (null / misaligned pointer, bad stride, rows < 0),
 * UNSUPPORTED (D), CUDA (launch failure). */
QPS_API qps_status qps_kv_quant_q8_0(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                             void* codes, void* scales, void* stream);

/* TQ3 encode [POLY, "What PolyKV is (reference)", "S2 — TurboQuant tier family",
 * "Phase-0 fork recon"].  Per row, in IEEE float32 with a fixed order: squares, a
 * halving-fold sum (t[i] += t[i+h] for h = D/2 .. 1), n = sqrt; u = FWHT(s .* x)
 * with butterflies (a+b, a-b) over stages h = 1, 2, ..., D/2; z = u / n; level index
 * = number of codebook thresholds <= z.  Stores the planes described above and
 * fp16(n).  A zero row stores zero planes and a zero norm.
 *   x       device, fp16 rows [rows][D], row stride x_row_stride (elements, >= D).
 *   signs   host, D/32 words: bit i of word i/32 set means s_i = -1.
 *   lo2     device, [rows][D/4] bytes;  hi1 device, [rows][D/8] bytes (4-byte aligned);
 *   norms   device, fp16 [rows].
 * D in {32, 64, 128, 256, 512}.  rows == 0 is a no-op.
 * Errors: INVALID_ARG, UNSUPPORTED (D), CUDA. */
QPS_API qps_status qps_kv_quant_tq3(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* lo2, void* hi1, void* norms,
                            void* stream);

/* TQ2 / TQ4 encode [POLY, "S2 — TurboQuant tier family"]: the TQ3 steps above with
 * the 4- or 16-level codebook
 * (qps_tq_codebook(2 or 4, ...)), storing one sign-magnitude field per element
 * (QPS_FMT_TQ2 / QPS_FMT_TQ4 above) and fp16(n).  A zero row stores zero fields and a
 * zero norm.
 *   x       device, fp16 rows [rows][D], row stride x_row_stride (elements, >= D).
 *   signs   host, D/32 words: bit i of word i/32 set means s_i = -1.
 *   codes   device, [rows][D/4] (TQ2) or [rows][D/2] (TQ4) bytes;
 *   norms   device, fp16 [rows]; 2-byte aligned (so is x).
 * D in {32, 64, 128, 256, 512}.  rows == 0 is a no-op.
 * Errors: INVALID_ARG, UNSUPPORTED (D), CUDA. */
QPS_API qps_status qps_kv_quant_tq2(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* codes, void* norms, void* stream);
QPS_API qps_status qps_kv_quant_tq4(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* codes, void* norms, void* stream);

/* TurboQuant encode at any tier and with either rotation form [POLY, "S2 —
 * TurboQuant tier family", "S2 perf-path Level B"]: R = diag(s2) blockdiag(H_G)
 * diag(s1) / sqrt(G).  Per row, in IEEE float32 with a fixed order: the norm as for
 * TQ3; u = FWHT stages h = 1 .. G/2 of s1 .* x; u = s2 .* u; z = (u * kappa) / n with
 * kappa = sqrtf(D / G) correctly rounded (1 when G = D); level index = number of
 * codebook thresholds <= z.  bits = 2, 3, 4 store the planes of QPS_FMT_TQ2 / TQ3 /
 * TQ4: plane0 = the data plane, plane1 = the TQ3 sign plane (4-byte aligned; NULL for
 * TQ2 / TQ4), norms = fp16 [rows].  signs1: host, D/32 words; signs2: host, D/32 words
 * or NULL; block: G (0 = D).  With signs2 = NULL and block = 0 this is
 * qps_kv_quant_tq2 / tq3 / tq4.  Errors: INVALID_ARG, UNSUPPORTED (D, bits), CUDA. */
QPS_API qps_status qps_kv_quant_tq_rot(int32_t bits, const void* x, int64_t rows, int32_t d,
                               int64_t x_row_stride, const uint32_t* signs1,
                               const uint32_t* signs2, int32_t block, void* plane0,
                               void* plane1, void* norms, void* stream);


/* A K or V cache (or one of its parts) as seen by the attention calls.  Row of
 * (token t, KV head h, batch entry b) = b*batch_stride + t*tok_stride + h*head_stride.
 * batch_stride == 0 means every batch entry reads the same rows (a shared prefix,
 * [POLY, "S1 — SharedKVPool"]); the attention then packs every batch entry's query
 * rows of a KV head into one tile so the shared rows are read once. */
typedef struct qps_kv_view {
  int32_t fmt;         /* qps_kv_format (TurboQuant: V, or K with V of the same tier) */
  int32_t reserved0;   /* must be 0 */
  const void* data;    /* device: F16 values | Q8_0 codes | TQ2/3/4 code plane; 16-byte aligned */
  const void* aux;     /* device: Q8_0 scales | TQ3 1-bit plane | TQ2/TQ4 norms; NULL for F16 */
  const void* aux2;    /* device: TQ3 norms; NULL otherwise */
  int64_t tok_stride;  /* rows between consecutive tokens (> 0) */
  int64_t head_stride; /* rows between consecutive KV heads (>= 0) */
  int64_t batch_stride;/* rows between consecutive batch entries; 0 = shared */
} qps_kv_view;

/* Arguments of one decode-attention part [RKV]: query rows attend key positions
 * [kv_begin, kv_end) of (k, v).  Logit s = scale * <q, k>; with softcap c > 0,
 * s <- c * tanh(s / c) before the softmax.  Query head h reads KV head h / (hq / hkv).
 * The positions are cut into n_split contiguous chunks (split-KV); each chunk yields a
 * normalised partial output and its natural-log LSE.  An empty chunk yields O = 0 and
 * lse = -inf.
 *
 * Output modes:
 *   o_parts != NULL : partials are written to part indices part_offset + s,
 *                     s in [0, n_split), of o_parts [parts][batch*hq][D] f32 and
 *                     lse_parts [parts][batch*hq] f32 (device); o / lse unused.
 *                     Merge them with qps_lse_combine.
 *   o_parts == NULL : the call merges its own chunks: o [batch*hq][D] f32 and
 *                     lse [batch*hq] f32 (device); needs `workspace` (device, 256-byte
 *                     aligned) of at least the size qps_attn_plan() reports.
 * Row index of (batch entry b, query head h) is b*hq + h in every output. */
typedef struct qps_attn_args {
  const void* q;          /* device, fp16 [batch][hq][D], 16-byte aligned */
  int64_t q_batch_stride; /* elements between batch entries (>= hq*D, multiple of 8) */
  int32_t batch, hq, hkv, d;
  qps_kv_view k, v;
  int64_t kv_begin, kv_end; /* 0 <= kv_begin <= kv_end < 2^31 - 64 (else UNSUPPORTED);
                               tokens of the views */
  float scale;
  float softcap;          /* <= 0: off */
  const uint32_t* v_signs;/* host, D/32 sign words of the cache's TurboQuant rotation;
                           required iff v.fmt is TQ2, TQ3 or TQ4 (a TurboQuant K uses
                           the same rotation, v_signs2 and v_block) */
  int32_t n_split;        /* > 0, or 0 = chosen by the library */
  int32_t part_offset;
  float* o_parts;
  float* lse_parts;
  float* o;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  /* Multi-query decode (verify batches) [POLY, "S2 perf-path — turbo-MMA verify
   * kernel"]: n_q query tokens per batch entry; 0 or 1 is single-token decode.  With
   * n_q > 1, q is fp16 [batch][n_q][hq][D] (q_batch_stride >= n_q*hq*D) and the output
   * row of (batch entry b, query token i, head h) is (b*n_q + i)*hq + h.
   * causal != 0: query token i sees only the view positions p <= q_pos + i (positions
   * counted like kv_begin / kv_end); a token that sees none of [kv_begin, kv_end) gets
   * O = 0 and lse = -inf.  n_q > 1 or causal needs the tensor-core path (see
   * qps_attn_path) and per-entry KV rows (batch_stride != 0 or batch == 1); in the
   * decode-step ring (qps_attn_decode_tail, qps_decode_step tails) q_pos is given in
   * the coordinates of the tiles' pos0 (qps_tile_desc), so that the newest positions of
   * a verify batch may lie in the tail.  Zero-initialised fields keep the single-token
   * behaviour. */
  int32_t n_q;
  int32_t causal;
  int64_t q_pos;
  /* The TurboQuant V rotation's second form [POLY, "S2 perf-path Level B" and its
   * head_dim-512 note]: R = diag(s2) blockdiag(H_G) diag(s1) / sqrt(G), s1 = v_signs.
   * v_signs2: host, D/32 words (bit set: -1) applied after the transform; NULL = none.
   * v_block: G, a power of two in [32, D] dividing D; 0 = D.  The V cache must have
   * been encoded with the same rotation (qps_kv_quant_tq_rot).  Zero-initialised
   * fields keep the first form R = H diag(s1) / sqrt(D). */
  const uint32_t* v_signs2;
  int32_t v_block;
  int32_t reserved1;      /* must be 0 */
} qps_attn_args;

/* Resolve the split count and the workspace the args need (host only, no launch):
 * the split-KV partition of [RKV] item S2 chosen for this GPU (no counterpart on the
 * pages for the choice itself).  n_split_out / workspace_bytes_out may be NULL.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA (the SM count of an automatic split). */
QPS_API qps_status qps_attn_plan(const qps_attn_args* a, int32_t* n_split_out,
                         size_t* workspace_bytes_out);

/* Which kernel the args select (host only): 1 = tensor-core path (every K / V plane
 * token-contiguous, tok_stride == 1, with 16-byte-aligned bases and head / batch
 * offsets), 0 = CUDA-core path (any other strides), negative = the args are invalid
 * (a qps_status, negated).  Both paths compute the same attention.  Library utility,
 * no counterpart on the pages.  Errors: as the negated return value. */
QPS_API int32_t qps_attn_path(const qps_attn_args* a);

/* Decode attention over device-resident KV (the window [0, wc), or any device part)
 * [RKV].  Supported: D in {64, 128, 256, 512}; K in {F16, Q8_0} with V in {F16, Q8_0, TQ2,
 * TQ3, TQ4}, or K and V in the same TurboQuant tier (TQ2 / TQ3 / TQ4: K is read in the
 * rotated domain against the rotated query, [POLY, "S2 perf-path Level B"]); hq a
 * multiple of hkv.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
QPS_API qps_status qps_attn_decode_window(const qps_attn_args* a, void* stream);

/* LSE combine [RKV, item S2]: M = max_t lse_t, w_t = exp(lse_t - M),
 * o = sum_t w_t O_t / sum_t w_t, lse = M + log sum_t w_t; parts with lse = -inf weigh
 * nothing; if all parts are empty, o = 0 and lse = -inf.
 *   o_parts   device, f32 [n_parts][rows][D];  lse_parts device, f32 [n_parts][rows].
 *   o         device, f32 [rows][D];           lse       device, f32 [rows].
 * n_parts >= 1, rows >= 0, D in {32, 64, 128, 256, 512, 1024}.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
QPS_API qps_status qps_lse_combine(const float* o_parts, const float* lse_parts, int32_t n_parts,
                           int64_t rows, int32_t d, float* o, float* lse, void* stream);

/* ---- Pinned host storage of the tail ------------------------------------------- */

/* Page-locked host memory for the tail ("F5 M7 — Rolling KV: position-windowed KV
 * residency", section "Storage layer": per-layer KV lives in pinned host memory
 * allocated with cudaHostAlloc(cudaHostAllocPortable)).  One large arena holding every
 * tile of the tail keeps the copy engine's reads on few, large page-locked regions.
 *   bytes  > 0;  flags: 0 = cudaHostAlloc portable | mapped, 1 = portable | mapped |
 *          write-combined, 2 = an anonymous mapping advised to use transparent huge
 *          pages, faulted in and registered with cudaHostRegister (portable | mapped);
 *          every allocation is mapped into the device's address space, so that the
 *          ring's copy kernel can read it (below);
 *   out    receives the host pointer (256-byte aligned), owned by the caller until
 *          qps_host_free.
 * Errors: INVALID_ARG, CUDA (allocation failure). */
QPS_API qps_status qps_host_alloc(size_t bytes, int32_t flags, void** out);

/* Free memory from qps_host_alloc (NULL is a no-op); the pinned tail of [RKV]
 * "Storage layer".  Errors: CUDA. */
QPS_API qps_status qps_host_free(void* p);

/* Copy `bytes` between device memory and qps_host_alloc memory with SM loads and stores
 * on `stream` (the ring's copy kernel; the copy engine is not used).  Exactly one of
 * dst / src lies inside one qps_host_alloc allocation and is reached through its device
 * mapping; the other is device memory.  Both 16-byte aligned; bytes == 0 is a no-op.
 * For a decode loop's per-step query upload and output readback: on GB300 hosts the
 * copy engine's transfers stall in bursts on some boxes (tens of ms) where SM loads of
 * the same memory do not (see qps_ring_set_copy_mode).  No counterpart on the pages.
 * Errors: INVALID_ARG (NULL, misaligned, neither or both in qps_host_alloc memory, the
 * host span leaving its allocation, or the other side not device memory), CUDA. */
QPS_API qps_status qps_copy_host(void* dst, const void* src, size_t bytes, void* stream);

/* ---- Tail-prefetch ring [RING] ------------------------------------------------ */

typedef struct qps_ring qps_ring;

/* [RING] Create a ring of n_slots (2..4) device staging slots of slot_bytes each on `device`,
 * a non-blocking copy stream and pre-created copy_done / compute_done events (timing
 * disabled).  The library owns these until qps_ring_destroy.  Makes `device` current.
 * Errors: INVALID_ARG, CUDA (allocation). */
QPS_API qps_status qps_ring_create(int32_t n_slots, size_t slot_bytes, int32_t device,
                           qps_ring** out);

/* [RING] Wait (bounded, 10 s) for the ring's copies, then free slots, events and the stream.
 * NULL is a no-op.  Errors: TIMEOUT (resources leaked rather than freed in use). */
QPS_API qps_status qps_ring_destroy(qps_ring* ring);

/* One tail tile: `tokens` consecutive positions of one layer's tail, stored in one
 * contiguous pinned-host range per plane, rows addressed inside the tile by
 * row = token * tok_stride + head * head_stride (the same for every plane of K and
 * V): token-major tiles use (hkv, 1), head-major tiles (1, padded tile length).  K
 * planes first (1 for F16, 2 for Q8_0, TQ2 and TQ4, 3 for TQ3, in data/aux/aux2 order), then V
 * planes.  The ring places each plane at the next 256-byte-aligned offset of the slot
 * (in that order); their total must fit in slot_bytes.  When the host planes already
 * sit at those offsets from the first K plane (a tail packed tile by tile), the whole
 * tile moves in one copy; otherwise each plane is its own copy.  Copies run on the
 * copy engine, or as the ring's copy kernel (64 small CTAs loading the mapped host
 * memory, on the copy stream) under QPS_RING_COPY_KERNEL (qps_ring_set_copy_mode). */
typedef struct qps_tile_desc {
  int32_t n_k_planes, n_v_planes;
  const void* host_k[3];
  size_t bytes_k[3];
  const void* host_v[3];
  size_t bytes_v[3];
  int64_t tokens;
  int64_t tok_stride;  /* rows; > 0 */
  int64_t head_stride; /* rows; >= 0 */
  int64_t pos0;        /* position of the tile's first token in the coordinates of the
                          attention's q_pos (the causal limit of a verify batch whose
                          newest positions lie in the tail); 0 when unused */
} qps_tile_desc;

/* [RING] How the ring moves tiles: QPS_RING_COPY_ENGINE (the default) uses the copy engine
 * (cudaMemcpyAsync) for every tile, leaving the SMs to the attention;
 * QPS_RING_COPY_KERNEL uses the ring's copy kernel for every tile whose planes lie in
 * qps_host_alloc memory (each on a 16-byte boundary) and the copy engine for the
 * others.  On GB300 hosts the copy engine's host-to-device transfers stall in bursts on
 * some boxes (single 1.3 ms transfers taking up to 50 ms) where SM loads of the same
 * memory do not; inside a decode step the copy kernel moves ~196 GB/s (the copy engine
 * 208 when it does not stall).  Takes effect from the next
 * qps_ring_begin_step.  Errors: STATE (invalid ring, open step), INVALID_ARG (mode). */
#define QPS_RING_COPY_ENGINE 0
#define QPS_RING_COPY_KERNEL 1
QPS_API qps_status qps_ring_set_copy_mode(qps_ring* ring, int32_t mode);

/* [RING] Start a step: copy the flat (layer, tile) schedule (host array, read during the
 * call) and enqueue the first n_slots tile copies on the copy stream; each copy
 * first waits for the compute_done event of the slot's previous user (which may
 * belong to the previous step).  Every host plane must be pinned.
 * Errors: INVALID_ARG (unpinned / null plane, tile larger than a slot), STATE (a step
 * is still open), CUDA. */
QPS_API qps_status qps_ring_begin_step(qps_ring* ring, const qps_tile_desc* tiles, int32_t n_tiles,
                               void* compute_stream);

/* Attend tile `tile_index` of the open step [RKV, RING].  Tiles must be consumed in
 * schedule order.  The compute stream waits for the slot's copy_done, the attention
 * runs on the slot (the k / v views' data pointers in `a` are ignored and replaced by
 * the slot's planes, their token / head strides by the tile's, their batch strides by
 * 0 (one tile serves every batch entry); their fmt is used; kv_begin / kv_end are
 * replaced by [0, tokens); with the causal limit, q_pos - pos0 of the tile), compute_done
 * is recorded, and the copy of tile tile_index + n_slots into the same slot is enqueued
 * behind it.  Output modes as for
 * qps_attn_decode_window.  Errors: STATE (out of order, no open step), INVALID_ARG,
 * UNSUPPORTED, CUDA. */
QPS_API qps_status qps_attn_decode_tail(qps_ring* ring, int32_t tile_index, const qps_attn_args* a,
                                void* compute_stream);

/* [RING] Close the step (every tile must have been consumed).  Does not wait for the
 * device.  Errors: STATE. */
QPS_API qps_status qps_ring_end_step(qps_ring* ring);

/* [RING] Wait until every copy and every tail attention issued by the ring has completed,
 * polling with a deadline of timeout_ms (never blocks longer).  Errors: TIMEOUT,
 * CUDA. */
QPS_API qps_status qps_ring_sync(qps_ring* ring, int32_t timeout_ms);

/* Guard regions of the ring's slots (failure detection; no counterpart on the pages:
 * the pages found their ring's write-after-read hazard only by byte-identity checks,
 * and this is the check for the other way a slot can be corrupted, a write outside
 * it).  Every slot is allocated with 256 guard bytes before and after it, filled with
 * a fixed per-slot pattern at qps_ring_create.  This call waits (bounded by
 * timeout_ms, as qps_ring_sync) until the ring's copies and tail attention are done,
 * reads both guards of every slot back (synchronous) and compares them with the
 * pattern.  bad_slot: host, may be NULL; set to -1, or to the first slot whose guard
 * changed.  The ring's device must be current.  Errors: INTERNAL (a guard changed:
 * something wrote outside its slot; the message names slot and side), TIMEOUT, STATE,
 * INVALID_ARG, CUDA. */
QPS_API qps_status qps_ring_check_guards(qps_ring* ring, int32_t timeout_ms, int32_t* bad_slot);

/* Device address and usable size (slot_bytes rounded up to 256) of ring slot `slot`,
 * for inspection and tests; the ring keeps owning the memory.  Library utility, no
 * counterpart on the pages.  data / bytes: host, either may be NULL.
 * Errors: STATE (invalid ring), INVALID_ARG (slot out of range). */
QPS_API qps_status qps_ring_slot(qps_ring* ring, int32_t slot, void** data, size_t* bytes);

/* Host-side fault injection for tests of the ring's error paths (no counterpart on the
 * pages; it exists so that a failed or late tile copy can be exercised without any GPU
 * fault).  Arms a one-shot fault on the next copy of schedule index tile_index, in
 * this or a later step:
 *   QPS_RING_FAULT_COPY_FAIL  the copy is not issued and the call issuing it
 *                             (qps_ring_begin_step, qps_attn_decode_tail or
 *                             qps_decode_step) returns QPS_ERR_CUDA, as a failed
 *                             cudaMemcpyAsync would; the step is closed;
 *   QPS_RING_FAULT_COPY_LATE  a host function that sleeps delay_ms (0..5000) runs on
 *                             the copy stream just before the copy, so the tile lands
 *                             late; the compute stream waits for it as for any tile;
 *   QPS_RING_FAULT_NONE       disarms.
 * Errors: STATE (invalid ring), INVALID_ARG (mode, tile_index < 0, delay_ms). */
#define QPS_RING_FAULT_NONE 0
#define QPS_RING_FAULT_COPY_FAIL 1
#define QPS_RING_FAULT_COPY_LATE 2
QPS_API qps_status qps_ring_inject_fault(qps_ring* ring, int32_t tile_index, int32_t mode, int32_t delay_ms);

/* ---- Native step runner -------------------------------------------------------- */

/* One layer of a decode step: device-resident parts (the window; for a shared-prefix
 * batch the prefix and the private suffixes), then `n_tiles` consecutive ring tiles
 * of this layer's tail attended with the `tail` template, then one LSE combine into
 * o / lse.  The runner assigns part indices: device part i takes the next n_split
 * indices after part i-1, then each tile its own n_split indices; the total must not
 * exceed parts_capacity.  The o_parts / lse_parts / part_offset / o / lse fields of
 * the per-part args are ignored (the runner sets them). */
typedef struct qps_layer_step {
  const qps_attn_args* device_parts; /* host array of n_device_parts args */
  int32_t n_device_parts;
  int32_t n_tiles;
  const qps_attn_args* tail;         /* host; required when n_tiles > 0 */
  float* o_parts;                    /* device, f32 [parts_capacity][batch*hq][D] */
  float* lse_parts;                  /* device, f32 [parts_capacity][batch*hq] */
  int32_t parts_capacity;
  float* o;                          /* device, f32 [batch*hq][D] */
  float* lse;                        /* device, f32 [batch*hq] */
  void* part_events[2];              /* optional cudaEvent_t pair (caller-created, may be
                                        NULL): recorded on the stream just before and just
                                        after this layer's device parts, for timing them */
} qps_layer_step;

/* Run one decode step over n_layers layers on `stream` [RKV, RING]: begin the ring
 * step with `tiles` (the concatenation of every layer's tiles, in layer order; ring
 * may be NULL when no layer has tiles), then for each layer its device parts, its
 * tiles and its combine, then close the ring step.  A layer's first device part runs
 * on `stream`; any further ones (e.g. the private suffixes beside a shared prefix) run
 * on library-owned side streams forked from `stream` by an event and joined back to it
 * before the layer's tiles, so independent parts overlap on the GPU.  Nothing waits for
 * the device.  Errors: as the calls it makes. */
QPS_API qps_status qps_decode_step(qps_ring* ring, const qps_tile_desc* tiles, int32_t n_tiles,
                           const qps_layer_step* layers, int32_t n_layers, void* stream);

/* qps_attn_decode_window in merged-output mode (o_parts == NULL, o / lse set) for
 * callers that cannot allocate device memory on the call path: code running where
 * cudaMalloc is forbidden or too costly (a serving loop whose device memory is owned
 * by an external pool, a latency-critical path that must not risk the synchronisation
 * an allocation can cause).  The pages describe no such entry point; it has no
 * counterpart there.  It allocates nothing: instead of a caller workspace, the split
 * partials live in a fixed 8 MiB file-scope device array that every GPU which loads
 * the library holds until the process exits.  `workspace` is ignored.
 *   - o / lse hold batch * n_q * hq rows ([rows][D] and [rows] f32, n_q >= 1).
 *   - Requests whose partials exceed the array (n_split * batch * n_q * hq * (D + 1)
 *     floats, plus alignment) fail with QPS_ERR_INVALID_ARG; pass a smaller n_split.
 *   - All calls on a device share the array and leave their partials in it (each call
 *     rewrites everything it reads); calls that overlap on the GPU race on it, so
 *     serialise them (one stream, or events between streams).
 *   - The first call on each device looks up the array's address and clears its error
 *     word (a synchronising step); make that first call before any stream capture.
 *   - A bounded in-kernel wait that gives up marks the array's error word instead of
 *     hanging and leaves the outputs invalid; this call does not read the word back.
 * Supported shapes and formats as qps_attn_decode_window (multi-query and causal decode
 * only on the tensor-core path).  Errors: INVALID_ARG (above, or o_parts set, or o / lse
 * NULL), UNSUPPORTED (n_q > 1 or causal with planes the tensor-core path cannot
 * stage), and otherwise as qps_attn_decode_window. */
QPS_API qps_status qps_attn_decode_window_noalloc(const qps_attn_args* a, void* stream);

/* Device-side status of the current device (failure detection; no counterpart on the
 * pages).  Kernels that wait on their own
 * asynchronous tile copies bound every wait; a wait that runs out sets a
 * library-owned device word instead of hanging, and the kernel returns early with
 * invalid outputs.  This call reads that word synchronously (it waits for the
 * device's pending work to reach it on the legacy stream) and clears it if `reset`.
 * Errors: INTERNAL (a bounds check of the checked build failed since the last reset;
 * see qps_build_checked), TIMEOUT (some wait gave up since the last reset), CUDA. */
QPS_API qps_status qps_device_status(int32_t reset);

/* The device error word and the record of the first bounded wait that gave up since
 * the last reset (failure detection; no counterpart on the pages), copied synchronously
 * into `words` (host, n words; words past the record are zeroed):
 *   [0] status bits (1: a wait gave up, 2: a bounds check failed), [1] number of waits
 *   that gave up, [2..4] that CTA's block index x / y / z, [5] its warp, [6] the warp's
 *   tile whose wait ran out, [7] tiles the warp had issued, [8] tiles the warp owns,
 *   [9] positions in the CTA's chunk, [10] ns the drain wait of that tile took,
 *   [11] 1 if the tile's copy completed during it, [12] ns of the last
 *   qps_selftest_bounded_wait's full bounded wait.
 * qps_device_status with reset clears all of it.  Errors: INVALID_ARG, CUDA. */
QPS_API qps_status qps_device_wait_record(uint32_t* words, int32_t n);

/* Self-test of the bounded waits above (no counterpart on the pages: it exists so that
 * the give-up path of a wait can be exercised on a GPU without any fault).  Enqueues on
 * `stream` one CTA of one warp that waits, with the same bounded wait the attention
 * kernels use on their tile copies, on a shared-memory barrier nothing ever arrives
 * on; once one second of the GPU's global timer has passed it sets the device error
 * word (and records the wait's duration, qps_device_wait_record word 12) and exits.  A
 * following qps_device_status then returns QPS_ERR_TIMEOUT (reset clears it).  The
 * call itself returns QPS_OK once the launch is enqueued.  Errors: CUDA. */
QPS_API qps_status qps_selftest_bounded_wait(void* stream);

/* 1 when this library is the bounds-checked build (libqps_checked.so, compiled with
 * QPS_CHECK_BOUNDS=1), else 0.  In that build every kernel tests each staged or
 * addressed access (tensor-map boxes and zero-filling copies into a tile stage, the
 * rows of a view, q, the partial outputs, the combine's outputs, the ring copy kernel's
 * writes into its slot) against the extent it must stay in; a failing access is
 * skipped and marks the device error word, which qps_device_status then reports as
 * QPS_ERR_INTERNAL.  A debug aid with no counterpart on the pages.  Never fails. */
QPS_API int32_t qps_build_checked(void);

/* Self-test of those bounds checks (no counterpart on the pages: it exercises the
 * checker's report without any out-of-bounds access).  Enqueues on `stream` one warp
 * that guards a store one past a 4-element shared array with the kernels' check; the
 * check fails, the store is skipped, and a following qps_device_status returns
 * QPS_ERR_INTERNAL (reset clears it).  Errors: UNSUPPORTED (not the checked build),
 * CUDA. */
QPS_API qps_status qps_selftest_bounds_check(void* stream);

/* Number of kernel launches the calling thread has issued through this library
 * since the last reset (reset if `reset` is non-zero).  Host only.  Library utility,
 * no counterpart on the pages.  Never fails. */
QPS_API int64_t qps_launch_count(int32_t reset);

/* ---- Residency and ring sizing policy (host arithmetic only) ------------------- */

/* Ring sizing [RKV, sections "Slot pool" and "Auto-adapt loop"]: the largest tile the
 * link moves while one layer's attention runs,
 *   tile_bytes_max = compute_ms_per_layer * 1e-3 * bw_eff_gbs * 1e9 * 0.8,
 * n_slots = clamp(floor(slot_budget_bytes / tile_bytes_max), 2, 4); a layer's tail is
 * cut into the fewest equal tiles of at most tile_bytes_max (tiles_per_layer, tile_bytes
 * rounded up; both 0 without a tail).  Inputs > 0 (per_layer_tail_bytes >= 0), finite;
 * any output pointer may be NULL.  Errors: INVALID_ARG. */
QPS_API qps_status qps_plan_ring(double compute_ms_per_layer, double bw_eff_gbs, double slot_budget_bytes,
                                 double per_layer_tail_bytes, int32_t* n_slots, int32_t* tiles_per_layer,
                                 double* tile_bytes, double* tile_bytes_max);

/* The negligible-drop tail band [TSTAR]: streaming a tail of B bytes slows a token by
 * (c_engage_ms + B / bw_eff) / t_resident_ms; the largest tail within target_drop is
 *   T* = (target_drop * t_resident_ms - c_engage_ms) * 1e-3 * bw_eff_gbs * 1e9,
 * reported as 0 when negative (never spill: compress instead).  t_resident_ms,
 * bw_eff_gbs > 0; c_engage_ms >= 0; 0 < target_drop < 1.  Errors: INVALID_ARG. */
QPS_API qps_status qps_tail_band(double t_resident_ms, double c_engage_ms, double bw_eff_gbs,
                                 double target_drop, double* t_star_bytes);

/* Storage tier choice [TSTAR, "The decision"]: the index of the first tier (ordered from
 * least to most compressing) whose KV bytes are <= budget_bytes + t_star_bytes, or the
 * last tier when none is (the rolling window then spills the rest).  n_tiers >= 1.
 * Errors: INVALID_ARG. */
QPS_API qps_status qps_choose_tier(const double* kv_bytes_per_tier, int32_t n_tiers, double budget_bytes,
                                   double t_star_bytes, int32_t* tier);

#ifdef __cplusplus
}
#endif

#endif /* QPS_H */
