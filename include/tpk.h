/*
 * tpk -- split-tier paged decode attention for GB300 (sm_103a).  C ABI.
 *
 * One decode step attends the G query rows of each KV head over a long paged
 * history held in two tiers (pages by their titles: "ActiveKV", section "The
 * idea"; "SYCL", sections "Attention that reads 8-bit history" and "A merge that
 * joins the tiers"; "model quantization", section "An 8-bit page format shaped
 * for its kernel"):
 *   - a recent tier of BF16 pages, attended exactly;
 *   - an older tier of 8-bit page records read directly, never expanded;
 *   - per-tier partials (output o, log-sum-exp lse) folded by an exact FP32 merge.
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership  The caller owns every buffer.  The library allocates no device
 *            memory; the multi-request call takes a caller-provided workspace.
 * Pointers   "dev" pointers are device memory of the current device; "host"
 *            pointers are read on the host before the call returns.  Device
 *            pointers must be 16-byte aligned.
 * Streams    Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *            legacy default stream).
 * Errors     Argument errors are detected on the host before any launch and
 *            returned as a status; nothing is launched then.  Launch failures
 *            map to TPK_ERR_CUDA.  Page-table entries outside the pool sizes
 *            given in tpk_shape are skipped by the kernels (that page then
 *            contributes nothing) and recorded in a device status word read by
 *            tpk_get_device_status.  The library never aborts or traps.
 *            tpk_last_error_string describes the last failure on this thread.
 * Layouts    BF16 pools:  [slot][kv_heads][64][256] bfloat16, K and V separate.
 *            8-bit pool:  record (slot, h) at byte (slot * kv_heads + h) * 35072.
 *            q:           [rows = kv_heads * group][256] bfloat16 (per request);
 *                         query row j belongs to KV head j / group.
 *            o:           float32 [rows][256], normalised (sum of weights 1).
 *            lse:         float32 [rows], natural log of sum exp(sm_scale q.k).
 * Empty      An empty token or page range yields lse = -inf and o = 0, the valid
 *            empty partial; a merge never reads the o of a -inf partial.
 * Contexts   Per device the library resolves once, on first use, the device
 *            addresses of its status word and static scratch, its kernels'
 *            shared-memory limits and its constant tables; they belong to the
 *            device's primary context.  Do not call cudaDeviceReset (or otherwise
 *            end that context) between calls of the library in one process.
 */
#ifndef TPK_H
#define TPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tpk_stream_t; /* identical to cudaStream_t */

typedef enum {
  TPK_OK = 0,
  TPK_ERR_INVALID = 1,     /* bad argument (null pointer, bad range, misalignment, too small buffer) */
  TPK_ERR_UNSUPPORTED = 2, /* shape outside what the kernels implement */
  TPK_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  TPK_ERR_BOUNDS = 4,      /* a kernel met a page-table entry outside the pool */
  TPK_ERR_NOMEM = 5,       /* a caller-provided buffer is smaller than required */
  TPK_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up */
  TPK_ERR_FORMAT = 7       /* a kernel met a malformed 13-bit record */
} tpk_status;

/* Which dot-product engine the decode kernels use. */
enum { TPK_IMPL_DEFAULT = 0, TPK_IMPL_SIMT = 1, TPK_IMPL_TENSOR = 2 };

/* Bytes of one 8-bit page-head record:
 *   u8   kc[64][256]   key codes, token-major          offset 0
 *   u8   vc[256][64]   value codes, channel-major      offset 16384
 *   f32  ks_chan[256]  key channel scale s_c           offset 32768
 *   f32  ks_tok[64]    key per-token factor r_t        offset 33792
 *   f32  vs_chan[256]  value channel scale u_c         offset 34048
 * Position swizzles (the format is shaped for the kernel that reads it):
 *   key code (t, c)   at byte t*256 + (c XOR 64*(t mod 2))
 *   value code (c, t) at byte c*64 + (t XOR 32*((c/2) mod 2))
 *   s_c               at float (c XOR 8*((c/32) mod 2))
 * A code c in [-127, 127] is stored as the byte c + 128 (offset binary), so
 * the tensor-core kernel widens it to f16 with one byte permute.
 * Dequantised: k_tc = kc_tc * s_c * r_t and v_tc = vc_tc * u_c. */
#define TPK_RECORD_BYTES 35072

typedef struct {
  int kv_heads;      /* H >= 1 */
  int group;         /* G query rows per KV head; must be 8 */
  int head_dim;      /* must be 256 */
  int page_tokens;   /* must be 64 */
  float sm_scale;    /* softmax scale; 0 selects 1/sqrt(head_dim) (the only value supported) */
  int impl;          /* TPK_IMPL_* */
  int64_t kv_slots;  /* slots in the BF16 pools (bounds for page_table entries); 0 = unchecked,
                        allowed only with TPK_IMPL_SIMT: the tensor-core kernel reads the BF16
                        pools through TMA tensor maps that need the pool size */
  int64_t rec_slots; /* slots in the 8-bit pool (bounds for page_table8 entries); 0 = unchecked */
  int int_query;     /* 0 (default): the 8-bit tier's QK uses the query in floating point.
                        1: the integer-query variant ("SYCL", "Attention that reads 8-bit
                        history": the integer query cache): per record and query row the
                        folded query q'_c = q_c s_c is coded as qi_c = rint(q'_c * (127 / m)),
                        m = max_c |q'_c| over the 256 channels, float32 steps with correctly
                        rounded divisions, half to even; the score is
                        (m / 127) * r_t * sum_c qi_c kc_tc, the sum exact.  This changes the
                        result (the query is coded to 8 bits); the exact tier is unaffected.
                        Tensor-core kernel only (TPK_IMPL_SIMT gives TPK_ERR_UNSUPPORTED). */
} tpk_shape;

const char* tpk_version(void);
const char* tpk_last_error_string(void);

/*
 * Page conversion ("model quantization", section "An 8-bit page format shaped for
 * its kernel").  For each of n_pages pages and each KV head h, read the BF16 page
 * (src_slots[i], h) of k_pool / v_pool and write record (dst_slots[i], h) of
 * rec_pool:
 *   key channel scale  s_c = sqrt(RMS_t k_tc), normalised by the geometric mean so
 *                      prod_c s_c = 1, clamped to [2^-14, 2^14], rounded to float32
 *                      with compensated rounding (the running log-error of the
 *                      product is kept nearest zero);
 *   key token factor   r_t = max_c |k_tc / s_c| / 127;
 *   value scale        u_c = max_t |v_tc| / 127;
 *   codes              kc = rint((k / s_c) / r_t), vc = rint(v / u_c), clamped to
 *                      +-127, with IEEE float32 divisions and half-to-even rint;
 *                      a zero factor gives zero codes.
 * src_slots, dst_slots: dev int32[n_pages].  k_pool, v_pool: dev BF16 pools.
 * rec_pool: dev, 16-byte aligned.  Pages may be converted in any order; distinct
 * dst_slots must not alias.  n_pages == 0 is a no-op.
 */
tpk_status tpk_kv_quantize_pages(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                                 const int32_t* src_slots, const int32_t* dst_slots, int n_pages,
                                 void* rec_pool, tpk_stream_t stream);

/*
 * As tpk_kv_quantize_pages, but with all three scale arrays given (dev float32
 * ks_chan[n_pages][H][256], ks_tok[n_pages][H][64], vs_chan[n_pages][H][256]);
 * only the codes are computed, and the given scales are copied into the records.
 * Used to check the codes bit for bit against a reference that fixed the scales.
 */
tpk_status tpk_kv_quantize_pages_given_scales(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                                              const int32_t* src_slots, const int32_t* dst_slots, int n_pages,
                                              const float* ks_chan, const float* ks_tok, const float* vs_chan,
                                              void* rec_pool, tpk_stream_t stream);

/*
 * Lossless 13-bit page format ("model quantization", section "A lossless tier
 * first": 13 bits per value, an 18.7 % saving, with a raw fallback when a plane
 * needs more than a 32-entry table).  A plane is one page-head's keys (or values):
 * 64 x 256 BF16 values, token-major.  A plane with at most 32 distinct exponent
 * fields is stored encoded (TPK_PACK13_PLANE_ENC bytes):
 *   u8 table[32]    the distinct exponent fields, ascending; unused entries 0  offset 0
 *   u8 sm[16384]    value i: (sign << 7) | 7-bit mantissa                     offset 32
 *   u8 lo4[8192]    table index bits 0-3: value 2j low nibble of byte j,
 *                   value 2j + 1 high nibble                                    offset 16416
 *   u8 hi1[2048]    table index bit 4 of value 8j + b in bit b of byte j        offset 24608
 * (8 + 5 bits per value), otherwise raw: the BF16 values (TPK_PACK13_PLANE_RAW
 * bytes).  A page-head record is a 16-byte header (u32 key-plane bytes, u32
 * value-plane bytes, two zero words) followed by the key plane and the value
 * plane; its size is 16 + both plane sizes, at most TPK_PACK13_RECORD_BYTES.
 */
#define TPK_PACK13_PLANE_ENC 26656
#define TPK_PACK13_PLANE_RAW 32768
#define TPK_PACK13_RECORD_BYTES 65552

/*
 * Pack n_pages BF16 pages into 13-bit records: page-head (src_slots[i], h) of
 * k_pool / v_pool -> record at pack_pool + (dst_slots[i] * H + h) *
 * TPK_PACK13_RECORD_BYTES (fixed-stride slots; the bytes of a slot past its
 * record's size are left unchanged).  src_slots, dst_slots: dev int32[n_pages];
 * pack_slots bounds dst_slots (0 = unchecked), shape->kv_slots bounds src_slots.
 * Pools 16-byte aligned.  An out-of-range slot skips that page-head and sets bit 0
 * of the device status word.  Lossless: tpk_kv_unpack13_pages restores every bit.
 */
tpk_status tpk_kv_pack13_pages(const tpk_shape* shape, const void* k_pool, const void* v_pool,
                               const int32_t* src_slots, const int32_t* dst_slots, int n_pages, void* pack_pool,
                               int64_t pack_slots, tpk_stream_t stream);

/*
 * Unpack n_pages pages of 13-bit records into BF16 pools: the record of page i,
 * KV head h starts rec_offsets[i * H + h] bytes into src (dev int64; 16-byte
 * aligned; fixed-stride slots or a compacted image alike) and is written to page
 * (dst_slots[i], h) of k_pool / v_pool.  src_bytes bounds the records (0 =
 * unchecked); shape->kv_slots bounds dst_slots.  A record whose header or extent
 * is invalid is skipped and sets bit 2 of the device status word (TPK_ERR_FORMAT
 * from tpk_get_device_status); an out-of-range slot sets bit 0.
 */
tpk_status tpk_kv_unpack13_pages(const tpk_shape* shape, const void* src, int64_t src_bytes,
                                 const int64_t* rec_offsets, const int32_t* dst_slots, int n_pages, void* k_pool,
                                 void* v_pool, tpk_stream_t stream);

/*
 * Exact-tier partial attention ("SYCL", section "A merge that joins the tiers":
 * paged decode with a log-sum-exp output).  For every KV head, the G query rows
 * attend BF16 tokens [tok_begin, tok_end) of one paged history whose token t lives
 * in slot page_table[t / 64], row t % 64.  The range is cut into num_splits
 * consecutive pieces on page boundaries (1 <= num_splits <= 4096); piece s writes
 * o_part[s] (dev float32 [num_splits][H*G][256]) and lse_part[s] (dev float32
 * [num_splits][H*G]).  A piece with no tokens writes the empty partial.
 * q: dev bf16 [H*G][256].  page_table: dev int32[ceil(tok_end / 64)].
 */
tpk_status tpk_decode_attn_exact(const tpk_shape* shape, const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* page_table, int tok_begin, int tok_end, int num_splits,
                                 float* o_part, float* lse_part, tpk_stream_t stream);

/*
 * 8-bit-tier partial attention ("SYCL", section "Attention that reads 8-bit
 * history").  As tpk_decode_attn_exact over pages [page_begin, page_end) of the
 * record pool, page p in slot page_table8[p] (dev int32[page_end]).  Keys enter
 * as q'_c = q_c * s_c folded once per page and score_t = r_t * sum_c q'_c kc_tc;
 * values accumulate on raw codes and are rescaled by u_c per page.
 */
tpk_status tpk_decode_attn_int8(const tpk_shape* shape, const void* q, const void* rec_pool,
                                const int32_t* page_table8, int page_begin, int page_end, int num_splits,
                                float* o_part, float* lse_part, tpk_stream_t stream);

/*
 * Log-sum-exp merge ("SYCL", section "A merge that joins the tiers"): fold
 * n_parts partials (dev o_parts [n_parts][rows][head_dim], lse_parts
 * [n_parts][rows]) into the accumulator (dev o_acc [rows][head_dim], lse_acc
 * [rows], read and written):
 *   lse = ln(exp(lse_acc) + sum_i exp(lse_i)),
 *   o   = exp(lse_acc - lse) o_acc + sum_i exp(lse_i - lse) o_i.
 * Partials with lse = -inf contribute nothing and their o is not read; a fresh
 * accumulator is (o = 0, lse = -inf).  The fold order is fixed (accumulator, then
 * parts in index order), so results are bit-reproducible.  head_dim must be 256.
 */
tpk_status tpk_merge_lse(int n_parts, int rows, int head_dim, const float* o_parts, const float* lse_parts,
                         float* o_acc, float* lse_acc, tpk_stream_t stream);

/*
 * Workspace bytes tpk_decode_hybrid_batched needs (partial results of the split
 * units, about 16 MiB; independent of the lengths).  The contents need no
 * initialisation.  tpk_workspace_init zero-fills a buffer (a convenience only).
 */
size_t tpk_hybrid_workspace_bytes(const tpk_shape* shape, int n_req);
tpk_status tpk_workspace_init(void* ws, size_t ws_bytes, tpk_stream_t stream);

/*
 * Multi-request hybrid decode ("SYCL", section "Exact tricks and a two-owner
 * decoder": requests in one launch, each with its own page metadata and its own
 * merge accumulator).  For each request b and KV head h: the exact partial over
 * its BF16 tokens [0, n_exact_tokens[b]) and the 8-bit partial over its pages
 * [0, n_int8_pages[b]), split across thread blocks of one decode launch, then
 * folded, in a fixed order, by a second small launch into o[b] (dev float32
 * [n_req][H*G][256]) and lse[b] (dev float32 [n_req][H*G]), which are
 * overwritten.
 *   q           dev bf16 [n_req][H*G][256]
 *   page_table  dev int32, flat; request b's exact-tier slots start at
 *               req_page_off[b] (host int32 [n_req + 1])
 *   page_table8 dev int32, flat; request b's 8-bit slots start at req_page_off8[b]
 *               (host int32 [n_req + 1])
 *   n_exact_tokens, n_int8_pages: host int32 [n_req]
 * The host arrays are read during the call (the split plan is built on the host
 * and passed by value to the kernels, so the call can be captured in a CUDA graph
 * once each device has seen one uncaptured call).
 * ws: dev workspace of at least tpk_hybrid_workspace_bytes(shape, n_req) bytes.
 * Calls sharing a workspace must not overlap on the GPU.
 */
tpk_status tpk_decode_hybrid_batched(const tpk_shape* shape, int n_req, const void* q, const void* k_pool,
                                     const void* v_pool, const void* rec_pool, const int32_t* page_table,
                                     const int32_t* req_page_off, const int32_t* n_exact_tokens,
                                     const int32_t* page_table8, const int32_t* req_page_off8,
                                     const int32_t* n_int8_pages, float* o, float* lse, void* ws, size_t ws_bytes,
                                     tpk_stream_t stream);

/*
 * The split plan tpk_decode_hybrid_batched makes, for inspection and sizing (host
 * only, no device work when resident_blocks > 0): for request b the thread blocks
 * (units) per KV head of the exact tier, splits_exact[b], and of the 8-bit tier,
 * splits_int8[b] (host int32 [n_req] each), and *n_units = H * the sum of both.
 * resident_blocks is the number of decode blocks the device holds at once (SMs x
 * blocks per SM), which sets the unit budget; 0 takes it from the current device
 * and shape->impl.  A segment gets at least one unit and at most one per page, an
 * empty request one empty exact unit; units carry about equal bytes.
 */
tpk_status tpk_hybrid_plan(const tpk_shape* shape, int n_req, const int32_t* n_exact_tokens,
                           const int32_t* n_int8_pages, int resident_blocks, int32_t* splits_exact,
                           int32_t* splits_int8, int32_t* n_units);

/*
 * Multi-request hybrid decode that allocates nothing and takes no workspace.
 * There is no counterpart in the pages this library follows: it exists for
 * callers that cannot hand the library device memory -- a plugin whose host
 * engine owns every device allocation and offers no way to ask for more, or a
 * runtime whose memory budget is fixed once serving starts.
 * Same arguments and results as tpk_decode_hybrid_batched, minus ws/ws_bytes.
 * Scratch: a file-scope device array of tpk_static_scratch_bytes() bytes
 * (16,842,752: the partials of the largest split plan, 2048 units), held by every
 * GPU that loads the library until the process exits.  A call whose plan needs
 * more fails with TPK_ERR_NOMEM.
 * The first call on a device resolves the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array and no state carries over between
 * calls that needs clearing, but calls that overlap on the GPU (for example on two
 * streams) race on it: serialise them.
 */
size_t tpk_static_scratch_bytes(void);
tpk_status tpk_decode_hybrid_batched_static(const tpk_shape* shape, int n_req, const void* q, const void* k_pool,
                                            const void* v_pool, const void* rec_pool, const int32_t* page_table,
                                            const int32_t* req_page_off, const int32_t* n_exact_tokens,
                                            const int32_t* page_table8, const int32_t* req_page_off8,
                                            const int32_t* n_int8_pages, float* o, float* lse,
                                            tpk_stream_t stream);

/*
 * Host-resident history staging ("ActiveKV", section on the host-authoritative KV
 * tier: pinned host memory holds every layer's history, the GPU a per-layer
 * staging working set of bounded size, filled by fenced asynchronous copies with
 * an explicit lifecycle, so a buffer is never reused while a copy or a kernel
 * still touches it).
 *
 * A stager owns one copy stream and two events per slot, created by
 * tpk_stager_create (not on the hot path); the slots are caller-owned device
 * buffers (16-byte aligned, slot_bytes each, on the device current at creation,
 * which must be current for every later call).  One host thread drives a stager.
 * Each slot cycles free -> staged -> acquired -> free:
 *   tpk_stager_stage    copies n_regions pinned host ranges (host_src[i], bytes[i])
 *                       to offsets slot_offset[i] of the next slot in round-robin
 *                       order, on the copy stream, after that slot's last release;
 *                       returns the slot index and its device address.  The host
 *                       ranges are read asynchronously: keep them valid until the
 *                       slot is acquired and the consumer has synchronised, or call
 *                       tpk_stager_sync.  Pageable sources are rejected.
 *   tpk_stager_acquire  makes `stream` wait for the slot's copies (call it right
 *                       before the work that reads the slot, so the copies of the
 *                       next layer overlap the current layer's decode).
 *   tpk_stager_release  records, on `stream`, that the work queued so far has
 *                       finished with the slot; the next staging into the slot
 *                       waits for it.
 * A call out of this order (staging into a slot that was not released, acquiring
 * a slot that is not staged, releasing one that is not acquired) returns
 * TPK_ERR_INVALID and changes nothing.  Not for use inside a stream capture.
 * tpk_stager_sync waits for every copy issued so far; tpk_stager_destroy waits for
 * them, then frees the stream and events (the slots stay the caller's).
 */
typedef struct tpk_stager tpk_stager;
tpk_status tpk_stager_create(int n_slots, void* const* slots, size_t slot_bytes, tpk_stager** out);
tpk_status tpk_stager_destroy(tpk_stager* stager);
tpk_status tpk_stager_stage(tpk_stager* stager, int n_regions, const void* const* host_src,
                            const size_t* slot_offset, const size_t* bytes, int* slot, void** slot_dev);
tpk_status tpk_stager_acquire(tpk_stager* stager, int slot, tpk_stream_t stream);
tpk_status tpk_stager_release(tpk_stager* stager, int slot, tpk_stream_t stream);
tpk_status tpk_stager_sync(tpk_stager* stager);
/*
 * Measured link behaviour ("Judge a representation by the bytes it stops
 * moving": a transfer model derived from the bus's measured behaviour): *ms =
 * the device time of the copies of the slot's latest staging, between events the
 * stager records on its copy stream right before the first and right after the
 * last of them (after the wait for the slot's release, so the copies alone).
 * Waits for those copies to finish; the slot's state is unchanged.
 */
tpk_status tpk_stager_copy_ms(tpk_stager* stager, int slot, float* ms);

/*
 * Incremental conversion and publication during decode ("ActiveKV": history
 * converted in the background and published to the decoder; "model
 * quantization": only whole pages older than the recent tokens become 8-bit).
 *
 * A tier manager follows the paged histories of n_req requests (page p of
 * request b in BF16 slot slots[p]; its record goes to the same slot of rec_pool),
 * in one layer or, with tpk_tiers_create_layers below, in several.  Each
 * tpk_tiers_step:
 *   1. publishes the pages whose conversion has finished (its event completed):
 *      they leave the exact tier and join the 8-bit tier;
 *   2. starts, on conv_stream, the conversion of every whole page that is now
 *      older than the recent_tokens newest tokens (after the work queued so far
 *      on decode_stream, which wrote those pages);
 *   3. fills `plan` with the step's tiers for tpk_decode_hybrid_batched: device
 *      page tables uploaded on decode_stream (use them on decode_stream), and host
 *      CSR offsets and counts valid until the next tpk_tiers_step.
 * A page is served exact until its conversion has finished, so a decode never
 * reads a record being written; the swap happens between steps.
 * tpk_tiers_update records request b's history after it grew: n_tokens and the
 * BF16 slots of its ceil(n_tokens / 64) pages (host array); a page converted or
 * being converted must keep its slot, and histories do not shrink.
 * Memory: dev_scratch (caller-owned, 256-byte aligned, tpk_tiers_device_bytes)
 * holds the page tables and conversion lists; two pinned host staging buffers
 * are allocated at creation and freed by tpk_tiers_destroy, which first waits
 * for the conversions in flight (tpk_tiers_sync waits without destroying).
 * One host thread drives a manager.
 */
typedef struct tpk_tiers tpk_tiers;
typedef struct {
  const int32_t* page_table;      /* dev: exact-tier slots, CSR by req_page_off */
  const int32_t* req_page_off;    /* host [n_req + 1] */
  const int32_t* n_exact_tokens;  /* host [n_req] */
  const int32_t* page_table8;     /* dev: 8-bit-tier slots, CSR by req_page_off8 */
  const int32_t* req_page_off8;   /* host [n_req + 1] */
  const int32_t* n_int8_pages;    /* host [n_req] */
  int pages_published;            /* pages that joined the 8-bit tier at this step */
  int pages_started;              /* conversions started at this step */
  int pages_converting;           /* conversions in flight after this step */
} tpk_tiers_plan;
size_t tpk_tiers_device_bytes(int n_req, int max_pages);
tpk_status tpk_tiers_create(const tpk_shape* shape, int n_req, int max_pages, int recent_tokens, const void* k_pool,
                            const void* v_pool, void* rec_pool, void* dev_scratch, size_t dev_scratch_bytes,
                            tpk_tiers** out);
tpk_status tpk_tiers_update(tpk_tiers* tiers, int b, int n_tokens, const int32_t* page_slots);
/*
 * The same manager over n_layers attention layers ("model quantization", "An
 * 8-bit page format shaped for its kernel": conversion only for pages fully
 * written in every layer, served exact until published).  The layers share the
 * requests' page tables: page p of request b lives in slot page_slots[p] of every
 * layer's pools (k_pools[l], v_pools[l]: dev BF16 pools; rec_pools[l]: dev record
 * pools; host arrays of n_layers pointers), so one plan serves every layer's
 * decode call.  A page becomes eligible once it is older than the recent window
 * and every layer has written it; its conversion runs in every layer on
 * conv_stream, and it is published -- in all layers at once -- at the first step
 * after one event recorded behind all of them.  host_rec_pools (NULL, or
 * n_layers pinned host record pools laid out like the device ones) receive a copy
 * of every converted record before that event ("ActiveKV", "The idea": host
 * memory holds the authoritative copy), so a published page's records are in the
 * host image too; the caller must not stage a page's records before it is
 * published.  tpk_tiers_create is this with one layer and no host pools.
 * tpk_tiers_update_layers records request b's history like tpk_tiers_update and
 * the tokens each layer has written so far (layer_written: host int32[n_layers],
 * each in [64 * (pages converted or being converted), n_tokens]); NULL, and
 * tpk_tiers_update, mean every layer has written all n_tokens.
 */
tpk_status tpk_tiers_create_layers(const tpk_shape* shape, int n_layers, int n_req, int max_pages, int recent_tokens,
                                   const void* const* k_pools, const void* const* v_pools, void* const* rec_pools,
                                   void* const* host_rec_pools, void* dev_scratch, size_t dev_scratch_bytes,
                                   tpk_tiers** out);
tpk_status tpk_tiers_update_layers(tpk_tiers* tiers, int b, int n_tokens, const int32_t* page_slots,
                                   const int32_t* layer_written);
tpk_status tpk_tiers_step(tpk_tiers* tiers, tpk_stream_t conv_stream, tpk_stream_t decode_stream,
                          tpk_tiers_plan* plan);
tpk_status tpk_tiers_sync(tpk_tiers* tiers);
tpk_status tpk_tiers_destroy(tpk_tiers* tiers);

/*
 * Measurement hook: while set, every decode-kernel launch of the library (the
 * partial calls and the decode launch of the multi-request call, not its fold) is
 * preceded by a record of `before` and followed by a record of `after` on the
 * launch stream (cudaEvent_t created with timing enabled), as external records, so
 * a CUDA graph captured meanwhile records them on each replay and
 * cudaEventElapsedTime(before, after) is the decode kernel's own duration.  Both
 * null clears it.  Process-wide; set it only while no other thread launches.
 */
tpk_status tpk_set_decode_timing_events(void* before, void* after);

/*
 * Test hook for the bounded device-side waits (no counterpart in the pages: it
 * lets a test make a wait run out without faulting or hanging the GPU).  Every
 * wait of a decode kernel on an mbarrier (for a copy to land, for a partner warp,
 * for a slot to be released) gives up after wait_limit_ns of wall time -- 0
 * restores the default of two seconds -- then sets bit 1 of the device status
 * word, lets the copies it issued land (each such wait bounded the same way) and
 * returns without writing its partial.  stall_unit >= 0 makes the tensor-core
 * decode kernel's thread block of that index (a split unit; tpk_hybrid_plan gives
 * the layout) leave its first history item unissued: no copy is made and nothing
 * arrives on that item's barrier, so the waits on it run out; the results of that
 * launch are then undefined.  -1 turns it off.  Process-wide, for the decode
 * launches made while it is set; set it only while no other thread launches.
 * Returns TPK_ERR_INVALID for stall_unit < -1 or a limit above 60 s.
 */
tpk_status tpk_set_test_wait(uint64_t wait_limit_ns, int stall_unit);

/*
 * Device status word: bit 0 = a page-table entry outside the pool was skipped,
 * bit 1 = a bounded device-side wait gave up, bit 2 = a malformed 13-bit record was
 * skipped.  Synchronises `stream`, stores the word in *flags and, if reset != 0,
 * clears it; returns TPK_ERR_TIMEOUT, TPK_ERR_BOUNDS or TPK_ERR_FORMAT (in that
 * order of precedence) when a bit is set.
 */
tpk_status tpk_get_device_status(int* flags, int reset, tpk_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TPK_H */
