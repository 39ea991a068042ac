/*
 * okvq.h - C ABI of libokvq: a 2/4-bit omni-modal KV cache with fused decode
 * attention for one GB300 (sm_103a).
 *
 * The operations follow "OmniKVQuant: KV Cache Quantization for Omni-LLMs"
 * (paperlayer.ai summary of arXiv 2609.11582):
 *   - section 2 METHOD, TurboQuant bullet: keys and values are rotated toward
 *     a Gaussian-like coordinate law with a randomized Hadamard transform, the
 *     magnitude is split from the direction, and a fixed codebook quantizes
 *     the rotated coordinates;
 *   - section 2, first OmniKVQuant bullet: rotated keys are min-max scaled
 *     within short groups of consecutive tokens, the group statistics are
 *     stored, and the shared fixed codebook quantizes the scaled values;
 *   - section 2, second OmniKVQuant bullet: values use one orthogonal
 *     eigenbasis rotation per modality;
 *   - section 1 INTRODUCTION, Implementation bullet: the fused decode unpacks
 *     the quantized cache inside attention without building a dense FP16
 *     cache, rotates the query once per head, and batches the inverse value
 *     rotations after attention aggregation.
 *
 * Readings of what the page leaves open (all fixed here, identically in the
 * library and in its test oracle):
 *   - head_dim is 128; the Hadamard matrix is Sylvester-ordered; the random
 *     signs are bit c of the SplitMix64 stream seeded with hadamard_seed
 *     (bit set -> -1), shared by every session, layer and head;
 *   - keys: k' = fp32(1/sqrt(d)) * FWHT(s o k) in fp32 with butterfly strides
 *     1, 2, ..., 64; groups of group_size consecutive tokens aligned to the
 *     absolute token index; per channel the group statistics are the min,
 *     stored fp16 rounded down, and the range max - min, stored fp16 rounded
 *     up, so [min, min + range] contains every member; u = (k'-min)/range in
 *     fp32 is coded to the nearest of the key levels
 *     lambda_j = (l_j - l_0) / (l_last - l_0); range 0 gives code 0;
 *     the keys of an incomplete trailing group stay in fp16 and are attended
 *     exactly until the group completes;
 *   - values: n = |v| stored fp16 (round to nearest even);
 *     w = sqrt(d) * R_m * v/n is coded to the nearest level l_j, with R_m the
 *     rotation of the token's modality (rows = basis vectors);
 *   - codebook: 2^bits ascending levels, rounded once to fp16 (the fp16
 *     values define the codebook); the default is the Lloyd-Max quantizer of
 *     N(0, 1); decisions compare fp32 values with fp32 midpoints of adjacent
 *     fp16 levels, a value equal to a midpoint taking the lower code;
 *   - decode attends every cached token of a session with one softmax
 *     (scale 1/sqrt(d)); query head h uses kv head h / (num_q_heads /
 *     num_kv_heads); the output is (sum_m R_m^T o_m) / l where o_m
 *     accumulates p_t * n_t * l(code_t) / sqrt(d) over tokens of modality m.
 *
 * Threading: a handle is not thread-safe; use one per thread or lock.
 * Streams: every call that takes a stream (a cudaStream_t passed as void*,
 * NULL = the legacy default stream) only enqueues work on it; caller buffers
 * must stay valid until that work has run.
 */
#ifndef OKVQ_H
#define OKVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct okvq_cache okvq_cache; /* opaque, owned by the library */

typedef enum {
  OKVQ_OK = 0,
  OKVQ_EINVAL = 1,    /* bad argument, shape or configuration; nothing was changed */
  OKVQ_ENOMEM = 2,    /* a device or host allocation failed */
  OKVQ_ECAPACITY = 3, /* the append would exceed max_tokens; nothing was written */
  OKVQ_ECUDA = 4,     /* a CUDA call or kernel launch failed */
  OKVQ_ESTATE = 5,    /* the device error word was set (e.g. a modality id out of range,
                         a bounded wait that gave up); see okvq_check_errors */
  OKVQ_ESCRATCH = 6   /* okvq_decode_static_scratch: the decode work list has more than
                         OKVQ_STATIC_SCRATCH_SEGMENTS segments; nothing was launched */
} okvq_status;

/* Key codec (okvq_config.key_codec). */
typedef enum {
  OKVQ_KEYS_GROUP_RANGE = 0, /* OmniKVQuant: per-group min-max of the rotated keys (section 2,
                                first OmniKVQuant bullet); the default */
  OKVQ_KEYS_TURBOQUANT = 1   /* TurboQuant, the pages' comparison point (section 2, TurboQuant
                                bullet): each key coded on arrival like a value, with the
                                shared randomized Hadamard rotation: n = |k| stored fp16,
                                w = sqrt(d) * (1/sqrt d) H D k/n coded with the value levels;
                                one global scale, no group statistics, no fp16 tail */
} okvq_key_codec;

typedef struct {
  int32_t num_sessions;   /* independent streams held by the cache, >= 1 */
  int32_t num_layers;     /* >= 1 */
  int32_t num_q_heads;    /* multiple of num_kv_heads, at most 8 query heads per kv head */
  int32_t num_kv_heads;   /* >= 1 */
  int32_t head_dim;       /* must be 128 */
  int32_t group_size;     /* key group size: 32 or 64 tokens */
  int32_t bits;           /* code width for keys and values: 2 or 4 */
  int32_t num_modalities; /* 1..3; modality ids are 0..num_modalities-1 */
  int64_t max_tokens;     /* per-session capacity, 1 .. 2^31 - 64; all storage is allocated by okvq_create */
  uint64_t hadamard_seed; /* seed of the shared random sign vector */
  const float *codebook;  /* host, 2^bits strictly ascending levels, or NULL for Lloyd-Max N(0,1);
                             copied at create */
  const float *value_rot; /* host, fp32 [num_layers][num_kv_heads][num_modalities][128][128],
                             row-major, row i = i-th basis vector; should be orthogonal (not
                             checked); copied at create. TurboQuant's single shared value
                             rotation is the Hadamard rotation (1/sqrt d) H D for every m. */
  int32_t key_codec;      /* okvq_key_codec; 0 (zero-initialised configs) = OmniKVQuant keys.
                             With OKVQ_KEYS_TURBOQUANT group_size is validated but unused. */
} okvq_config;

/* Allocate a cache. Validates cfg (OKVQ_EINVAL), allocates device storage
 * (OKVQ_ENOMEM) and uploads the codebook and rotations on `stream`, then
 * synchronizes it. On success *out owns everything until okvq_free. */
okvq_status okvq_create(const okvq_config *cfg, void *stream, okvq_cache **out);

/* Release a cache and all its device memory (synchronizes the device). NULL is a no-op. */
void okvq_free(okvq_cache *h);

/* Append num_tokens tokens to `session` (section 2: values are quantized at
 * once; each key group is quantized when its last token arrives).
 *   k, v      device fp16 [num_tokens][num_layers][num_kv_heads][128], token-major,
 *             16-byte aligned (the value rows are copied in 16-byte pieces)
 *   modality  device uint8 [num_tokens], each < num_modalities (checked on the
 *             device: a bad id sets the error word and is stored as modality 0)
 * Shapes, alignment and capacity are checked on the host before any launch
 * (OKVQ_EINVAL / OKVQ_ECAPACITY, state unchanged). num_tokens == 0 is a no-op.
 * Two kernel grids, asynchronous: the values on `stream`, the keys on a stream
 * owned by the handle that waits for `stream` before it starts (an event) and
 * that `stream` waits for afterwards (another event), so work issued on `stream`
 * after the call sees the whole append. Appends of one handle must be ordered
 * (one host thread). */
okvq_status okvq_append_chunk(okvq_cache *h, int32_t session, const void *k, const void *v,
                              const uint8_t *modality, int32_t num_tokens, void *stream);

/* One decode step for every session and layer (section 1, Implementation):
 *   q    device fp16 [num_sessions][num_layers][num_q_heads][128], 16-byte
 *        aligned (each segment's queries arrive by bulk copy); OKVQ_EINVAL otherwise
 *   out  device fp16 [num_sessions][num_layers][num_q_heads][128]
 * An empty session yields zeros. Two kernel launches (split-K fused
 * attention, then the merge + inverse value rotations), asynchronous on
 * `stream`.
 * Work list: the first decode after appends (or an eviction or compaction)
 * changed the lengths plans the split on the host and uploads it on `stream`
 * from one of two page-locked staging buffers used in turn; the call waits
 * only for the upload made from the same buffer two rebuilds earlier (in an
 * append-then-decode loop that upload has long finished). That upload reads
 * host memory when it runs, so such a first decode is not for stream capture;
 * decodes with unchanged lengths upload nothing. The device copy of the work
 * list is one per handle: calls on one handle must be ordered on the device
 * (one stream, or ordered by the caller). */
okvq_status okvq_decode(okvq_cache *h, const void *q, void *out, void *stream);

/* Capacity, in work-list segments, of the static scratch array used by
 * okvq_decode_static_scratch: 512 segments of 8 heads x (2 + 3*128) floats,
 * 6,324,224 bytes of device memory reserved when the library's device code is
 * loaded on a device. A decode's work list has at most
 * (SM count + num_sessions*num_layers*num_kv_heads) segments. */
#define OKVQ_STATIC_SCRATCH_SEGMENTS 512

/* okvq_decode without per-call scratch memory of its own. The OmniKVQuant
 * page has no counterpart of this call: it is an engineering variant of
 * okvq_decode (same arguments, same kernels, same results) whose split-K
 * partials go to one file-scope device array of OKVQ_STATIC_SCRATCH_SEGMENTS
 * segments instead of the handle's partials buffer, and which never creates
 * CUDA events (okvq_profile_* record okvq_decode only). It allocates nothing:
 * no cudaMalloc, cudaFree, event or library allocation.
 * It is meant for callers that must not allocate device memory, or let a
 * library allocate for them, during the call. One example is a serving loop
 * whose device memory is handed out by its own allocator or a fixed budget.
 * Another is a latency-critical decode step that must keep the device
 * allocator, and the synchronisation cudaFree implies, out of its path.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress with the handle's device made current, then the
 * previous device restored), once per device for the process; OKVQ_ECUDA if
 * that fails (retried on the next call). Make that first call before any
 * stream capture.
 * Sharing: every call, from every handle on a device, uses the same array.
 * It keeps the last call's contents; nothing in it needs to start at zero,
 * because each call writes every partial it reads. Calls whose work overlaps
 * on the device (different streams, or threads without ordering) race on the
 * array and give undefined results: order them on one stream or serialise them.
 * Errors: OKVQ_EINVAL for NULL arguments; OKVQ_ESCRATCH, with nothing launched,
 * when the current work list has more than OKVQ_STATIC_SCRATCH_SEGMENTS
 * segments (the work list itself, shared with okvq_decode, may have been
 * rebuilt and uploaded on `stream`); otherwise as okvq_decode. */
okvq_status okvq_decode_static_scratch(okvq_cache *h, const void *q, void *out, void *stream);

/* okvq_decode on HOST buffers: brings the queries (host, same layout as
 * okvq_decode's q) into the handle's device staging, decodes, and delivers the
 * outputs to `out_host`, all asynchronously on `stream` (the host buffers must
 * stay valid, and `out_host` unread, until the stream reaches that point).
 * Page-locked host memory (cudaHostAlloc, cudaHostRegister, a pinned torch
 * tensor; checked with cudaPointerGetAttributes on every call):
 *  - queries (16-byte aligned): a small kernel on `stream` reads them through
 *    their mapped device address and writes the staging once every earlier
 *    kernel on `stream` has completed; it runs, like the decode, as a programmatic
 *    dependent of the kernel before it, so the decode's prologue still overlaps
 *    the previous call's merge;
 *  - outputs: the merge kernel stores them into `out_host` directly, with no copy
 *    after the decode.
 * Pageable memory: the queries are uploaded (synchronously with respect to the
 * host) on a copy stream owned by the handle, into one of two staging slots, so
 * the upload overlaps the decode a previous call left on `stream`; `stream` waits
 * for it. The outputs go through device staging and a copy on `stream`. The
 * call's effects are complete when `stream` reaches that point. Staging
 * (4 x S*L*Hq*128 fp16), the copy stream and its events are created by
 * okvq_create; calls on one handle must be ordered (one host thread). Errors as
 * okvq_decode. */
okvq_status okvq_decode_host(okvq_cache *h, const void *q_host, void *out_host, void *stream);

/* Decode with far-memory pseudo tokens ("ProtoKV: Streaming Video Understanding
 * under Delayed Query with Summary-State Memory", section 3.3 Eq. (2), Appendix
 * A.3 Eq. (4) and Algorithm 4): one softmax per query head over the cache (the
 * near window, bias 0, evicted tokens skipped) and P = num_prototypes x
 * S = tokens_per_prototype pseudo tokens per (session, layer, kv head) that the
 * caller synthesized (prototype centre plus decoded residual modes; the
 * synthesis itself is the caller's). Pseudo token j belongs to prototype j / S,
 * whose mass n adds log n to its logit q.k/sqrt(d); prototypes with n = 0 are
 * inactive and skipped. Layouts (device, row-major):
 *   q, out     as okvq_decode
 *   far_k      fp16 [S][L][Hkv][P*S][128]  pseudo keys, the caller's key basis
 *              (the one okvq_append_chunk receives keys in), 16-byte aligned
 *   far_v      fp16 [S][L][Hkv][P*S][128]  pseudo values, the original value basis, 16-byte aligned
 *   far_mass   fp32 [S][L][Hkv][P]         n >= 0
 * Launches the near-window decode, one far-memory kernel and the merge on
 * `stream`; nothing is allocated (the far partials are reserved by okvq_create).
 * P = 0 gives okvq_decode's result. A unit with no live near token and no
 * active prototype decodes to zeros. OKVQ_EINVAL for NULL or misaligned
 * pointers, P < 0, S < 1 or P*S > 2^30. With profiling on, okvq_profile_read's
 * first time covers the near-window and far-memory kernels together. */
okvq_status okvq_decode_pseudo(okvq_cache *h, const void *q, const void *far_k, const void *far_v,
                               const float *far_mass, int32_t num_prototypes, int32_t tokens_per_prototype,
                               void *out, void *stream);

/* Device pointers passed to okvq_append_chunk, okvq_decode, okvq_decode_static_scratch,
 * okvq_decode_pseudo and okvq_calibrate_rotations are checked with
 * cudaPointerGetAttributes: host memory (pageable or pinned) or another device's
 * memory gives OKVQ_EINVAL with nothing launched. A handle remembers the last 8
 * pointers it accepted, so a loop over fixed buffers pays the query once. */

/* Number of token slots of `session`: its physical span, holes included (the
 * next append lands at this index). */
okvq_status okvq_length(const okvq_cache *h, int32_t session, int64_t *tokens);

/* Slots of `session` that hold a token that was not evicted. */
okvq_status okvq_live_length(const okvq_cache *h, int32_t session, int64_t *tokens);

/* ---- eviction and compaction ("OmniTide: Co-Designing Algorithms and Systems
 * for Efficient On-Device Omni-LLM Streaming", section 5.2 Applying the
 * retention plan and section 6.2 Selective and efficient KV migration) ---- */

/* Delete token slots of `session` in every (layer, kv head): `ranges` is a HOST
 * array of num_ranges [begin, end) pairs of slot indices, 0 <= begin <= end <=
 * okvq_length. Deleted tokens stay in their slots as holes that okvq_decode
 * skips (they take no part in the softmax); a session whose every token is
 * deleted decodes to zeros. Deleting a deleted slot again is allowed. Key group
 * statistics are not recomputed: the survivors of a group keep its statistics,
 * and a group still open when some of its members are deleted is completed by
 * later appends over all its members. Logical positions (RoPE) are the caller's.
 * Asynchronous on `stream` (one small copy and one kernel); the slot count is
 * unchanged. OKVQ_EINVAL for a bad session, a range outside [0, length] or
 * end < begin (nothing changes). */
okvq_status okvq_evict(okvq_cache *h, int32_t session, const int64_t *ranges, int32_t num_ranges, void *stream);

/* Tokens that compaction moves as one unit: the key group size, or 16 (one tile)
 * with OKVQ_KEYS_TURBOQUANT. A key group moves whole because its statistics
 * serve all its members. */
okvq_status okvq_compaction_granule(const okvq_cache *h, int32_t *tokens);

/* The ordered-suffix migration plan, on the host (no handle, no GPU): with
 * `dead` a HOST array of `length` bytes (nonzero = deleted) and granules of
 * `granule` slots (16, 32 or 64), scan suffix starts s (multiples of the
 * granule) from the end backward; packing the suffix's granules that still hold
 * a live token to s, s + granule, ... in their order gives a new length T'; the
 * first (shortest) suffix with ceil(length/64) - ceil(T'/64) >= min_pages_saved
 * (>= 1) is the plan. Outputs: *suffix_begin = s (-1 when no suffix saves enough:
 * nothing moves), *new_length = T' (length when none), *num_moves = granules whose
 * slot changes. OKVQ_EINVAL for bad sizes or NULL pointers. */
okvq_status okvq_plan_compaction(const uint8_t *dead, int64_t length, int32_t granule, int32_t min_pages_saved,
                                 int64_t *suffix_begin, int64_t *new_length, int32_t *num_moves);

/* The decode's split of the work over CTAs, on the host (no handle, no GPU):
 * the pages of units 0..units-1 (unit_pages[u] >= 0 each, HOST array), in
 * order, are cut into at most max_ctas contiguous ranges, one per CTA, and each
 * range into segments at unit boundaries (one split-K partial each). A page
 * costs 1 and a segment segment_cost more; the split minimises the largest
 * CTA cost (the smallest budget with which a greedy walk covers every page,
 * found by bisection), and no segment is empty. okvq_decode's own split
 * (okvq_plan_decode_work, below) starts from this one with segment_cost 48 (a
 * segment's query rotation, its empty page ring at the start and its cross-warp
 * merge at the end cost about that many pages in this model).
 * Outputs: segments [*num_segments][3] = unit, first page, end page (caller
 * room for units + max_ctas segments); cta_first [*num_ctas + 1] = first
 * segment of each CTA, then *num_segments (caller room for max_ctas + 1).
 * No pages: *num_ctas = *num_segments = 0. OKVQ_EINVAL for NULL pointers,
 * units < 0, max_ctas < 1, segment_cost < 0 or a count outside [0, 2^31). */
okvq_status okvq_plan_decode(const int64_t *unit_pages, int64_t units, int32_t max_ctas, int32_t segment_cost,
                             int32_t *segments, int32_t *cta_first, int32_t *num_ctas, int32_t *num_segments);

/* The split okvq_decode itself uses (host only; no handle, no GPU). A decode CTA's
 * warps (12 at bits 2, 8 at bits 4) take its pages in turn, so a segment of n
 * pages costs ceil(n / warps) whole rows. Two candidates: the contiguous split of
 * okvq_plan_decode with segment_cost 48, and a row-aligned split, in which every
 * unit is cut into pieces of R whole rows, one CTA each, and each unit's last pages
 * (fewer than a piece) go, costliest first, to the least loaded CTA holding no
 * piece. Under the model "a segment costs 12 + warps * ceil(n / warps) pages" the
 * row-aligned split is taken when its costliest CTA is at least one row cheaper
 * (the smallest R that fits, trying up to 64 values and skipping those whose cost
 * fills more than 99.8 % of the CTAs: the greedy packing needs slack). Example: 72 units of 512 pages
 * on 152 CTAs at bits 2: 144 CTAs take 252 pages (21 rows, not 22) and 8 CTAs take
 * nine 8-page remainders each. A unit's segments get consecutive partial slots in
 * page order. Inputs as okvq_plan_decode, and bits (2 or 4). Outputs: segments
 * [*num_segments][4] = unit, first page, end page, partial slot (caller room for
 * units + max_ctas + 1 segments), in CTA order; cta_first [*num_ctas + 1] = first
 * segment of each CTA, then *num_segments (room for max_ctas + 1); unit_first
 * [units + 1] = first partial slot of each unit, then *num_segments. No pages:
 * *num_ctas = *num_segments = 0. OKVQ_EINVAL for NULL pointers, units < 0,
 * max_ctas < 1, bits other than 2 or 4, or a count outside [0, 2^31). */
okvq_status okvq_plan_decode_work(const int64_t *unit_pages, int64_t units, int32_t max_ctas, int32_t bits,
                                  int32_t *segments, int32_t *cta_first, int32_t *unit_first, int32_t *num_ctas,
                                  int32_t *num_segments);

/* Plan (as okvq_plan_compaction, with the handle's granule and its deletions)
 * and apply the ordered-suffix compaction of `session`: the moved granules'
 * codes, statistics, norms, modality ids, masks and deletion bits are gathered
 * into a scratch buffer, then written to their new slots (so no move overwrites
 * another's source); the session's slot count becomes *new_length. The fp16
 * trailing keys of an open group need no move: a granule moves by whole groups,
 * so every token keeps its place within its group. The slot of a token that did
 * not move is unchanged; a moved token's new slot is its old slot minus the
 * granules removed before it. Outputs (host, may be NULL): *new_length,
 * *moved_granules (0 when no suffix saves min_pages_saved pages: nothing changes).
 * Asynchronous on `stream`; nothing is allocated (okvq_create reserves the
 * scratch: room for every granule of one session, at most 64 MB, and larger
 * plans run in batches). OKVQ_EINVAL for a bad session or min_pages_saved < 1. */
okvq_status okvq_compact(okvq_cache *h, int32_t session, int32_t min_pages_saved, int64_t *new_length,
                         int32_t *moved_granules, void *stream);

/* Copy the stored state of `session` to host memory in the canonical layout
 * (synchronizes the device). With host_buf == NULL only *bytes is set. With
 * T tokens, Tf = T - T % group_size, B = 128*bits/8, the buffer holds, in order:
 *   kcodes  uint8 [L][Hkv][Tf][B]   channel c at byte c*bits/8, bit (c*bits)%8
 *   kstats  fp16  [L][Hkv][Tf/group_size][2][128]   (min, range)
 *   ktail   fp16  [L][Hkv][T-Tf][128]               (unquantized trailing keys)
 *   vcodes  uint8 [L][Hkv][T][B]
 *   vnorm   fp16  [L][Hkv][T]
 *   mod     uint8 [T]
 *   dead    uint8 [L][Hkv][T]   1 where the token was evicted (read from each
 *                               (layer, kv head)'s own pages)
 * With OKVQ_KEYS_TURBOQUANT every key is quantized (Tf = T) and kstats/ktail
 * are replaced by knorm fp16 [L][Hkv][T] (|k|).
 * *bytes must hold the buffer size on entry (OKVQ_EINVAL if too small). */
okvq_status okvq_export_state(okvq_cache *h, int32_t session, void *host_buf, size_t *bytes);

/* The fp16-rounded value levels in use (2^bits floats) and the key levels
 * lambda_j (2^bits floats); either pointer may be NULL. */
okvq_status okvq_codebook(const okvq_cache *h, float *levels, float *key_levels);

/* Synchronize `stream`, read and clear the device error word. OKVQ_OK if it
 * was clear, OKVQ_ESTATE otherwise (*word, if non-NULL, receives its bits:
 * 1 = bad modality id, 2 = a bounded wait gave up). */
okvq_status okvq_check_errors(okvq_cache *h, void *stream, uint32_t *word);

/* Per-kernel timing with CUDA events recorded around each launch of
 * okvq_decode on its stream. enable != 0 clears and starts the record.
 * okvq_profile_read synchronizes, then returns the number of decode calls
 * recorded (at most `cap`) and their split-K kernel and merge kernel times
 * in milliseconds. */
okvq_status okvq_profile_enable(okvq_cache *h, int enable);
okvq_status okvq_profile_read(okvq_cache *h, float *split_ms, float *merge_ms, int32_t cap, int32_t *count);

/* Calibrate the per-modality value rotations (section 2, second OmniKVQuant
 * bullet: directions weighted by their contribution to attention outputs, one
 * covariance per modality, its eigenbasis as the rotation). For every
 * (layer, kv head) and modality m, over the calibration tokens of modality m:
 *   C_m = sum_t a_t (v_t - mu_m)(v_t - mu_m)^T / sum_t a_t,  mu_m the a-weighted mean,
 * and R_m = its eigenvectors as rows, in descending eigenvalue order, each row
 * signed so that its largest-magnitude entry is positive (fp32 cyclic Jacobi).
 * A modality with fewer than two tokens, or zero total weight, gets the identity
 * (eigenvalues 0). Tokens whose modality id is >= num_modalities are ignored.
 *   v         device fp16 [num_tokens][num_layers][num_kv_heads][128], token-major
 *   modality  device uint8 [num_tokens]
 *   weight    device fp32 [num_tokens][num_layers][num_kv_heads] (the a_t, >= 0),
 *             or NULL for all ones (the plain covariance)
 *   rot_out   device fp32 [num_layers][num_kv_heads][num_modalities][128][128]: the
 *             value_rot layout of okvq_config (copy it to the host for okvq_create)
 *   eig_out   device fp32 [num_layers][num_kv_heads][num_modalities][128], or NULL
 *   sweeps_out device int32 [num_layers][num_kv_heads][num_modalities], or NULL: the
 *             Jacobi sweeps run (the last one rotated nothing); negated when 30 sweeps
 *             did not converge (the basis is then the last iterate); 0 for identity
 * OKVQ_EINVAL for bad sizes or NULL required pointers; one kernel launch,
 * asynchronous on `stream`; nothing is allocated. */
okvq_status okvq_calibrate_rotations(int32_t num_layers, int32_t num_kv_heads, int32_t num_modalities,
                                     const void *v, const uint8_t *modality, const float *weight,
                                     int32_t num_tokens, float *rot_out, float *eig_out, int32_t *sweeps_out,
                                     void *stream);

/* Test hook: the n-th device allocation of the library from now on (n = 0: the
 * next one) fails as if the device were out of memory, so that the error paths of
 * okvq_create can be exercised without exhausting a GPU; n < 0 turns it off.
 * Process-wide; not for production use. */
okvq_status okvq_test_fail_alloc(int64_t n);

/* Static description of a status code. */
const char *okvq_status_string(okvq_status s);

#ifdef __cplusplus
}
#endif
#endif /* OKVQ_H */
