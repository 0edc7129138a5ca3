/*
 * kvd.h -- C ABI of the GB300 KV-cache decode-attention library.
 *
 * One process, one GPU (sm_103a).  Every device buffer is allocated by the
 * caller (by any CUDA allocator) and passed in as a plain pointer;
 * the library computes the sizes, never allocates device memory and keeps
 * no global state beyond caches of per-device kernel attributes and
 * occupancy (and the scratch array of decode_attention_static).  Every call is asynchronous on the caller's CUDA stream
 * (`stream` is a cudaStream_t passed as void*, NULL = legacy default
 * stream) unless its comment says otherwise.
 *
 * Errors.  Every entry point returns a kvd_status.  Arguments are checked
 * on the host BEFORE anything is launched or mutated: a call that returns
 * an error other than KVD_ECUDA has changed neither the cache contents nor
 * the host-mirrored cursors.  KVD_ECUDA reports a failed CUDA launch or
 * copy (the stream is then in an unknown state).  Kernels never trap: an
 * inconsistency they detect (a bound violated by corrupt metadata, a wait
 * that timed out) sets a device error word that kvd_layer_device_error /
 * rswa_device_error read back after the caller synchronises.
 *
 * Sources (page title, then the item on the page):
 *   cortiq  = docs.rs cortiq-engine 0.8.49, src/cortiq_engine/kv_cache.rs
 *   rswa    = franken_ocr 0.8.0, src/native_engine/rswa.rs
 */
#ifndef KVD_H
#define KVD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVD_API __attribute__((visibility("default")))
#else
#define KVD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Storage mode of one layer (cortiq KvMode): KVD_F32 stores f32 K and V;
 * KVD_Q8 (q8_2f) stores int8 K with one f32 scale per 32 channels and int8
 * V with one f32 scale per row, both against per-channel fields frozen
 * after 64 rows; KVD_Q8K quantises K only, KVD_Q8V V only. */
typedef enum { KVD_F32 = 0, KVD_Q8 = 1, KVD_Q8K = 2, KVD_Q8V = 3 } kvd_mode;

typedef enum {
    KVD_OK = 0,
    KVD_EINVAL = -1,    /* malformed argument (null pointer, bad size/shape) */
    KVD_ECAPACITY = -2, /* a sequence or ring would exceed its capacity      */
    KVD_ESTATE = -3,    /* call not valid in the current state (no prefill)  */
    KVD_EEMPTY = -4,    /* empty attention key set                           */
    KVD_ECUDA = -5,     /* a CUDA launch or copy failed                      */
    KVD_EDEVICE = -6    /* the device error word was set by a kernel         */
} kvd_status;

/* Device buffers of one layer, indexed by these slots in the size array of
 * kvd_layer_bytes and the pointer array of kvd_layer_init.  A slot whose
 * size is 0 for the chosen mode takes a NULL pointer. */
enum {
    KVD_BUF_K = 0,    /* f32  K rows            (KVD_F32, KVD_Q8V)          */
    KVD_BUF_V = 1,    /* f32  V rows            (KVD_F32, KVD_Q8K)          */
    KVD_BUF_KQ = 2,   /* int8 K codes           (KVD_Q8, KVD_Q8K)           */
    KVD_BUF_VQ = 3,   /* int8 V codes           (KVD_Q8, KVD_Q8V)           */
    KVD_BUF_KS = 4,   /* f32  K scale per 32 ch (KVD_Q8, KVD_Q8K)           */
    KVD_BUF_VS = 5,   /* f32  V scale per row   (KVD_Q8, KVD_Q8V)           */
    KVD_BUF_KCOL = 6, /* f32  K channel field [n_seq][n_live][hd]           */
    KVD_BUF_VCOL = 7, /* f32  V channel field [n_seq][n_live][hd]           */
    KVD_BUF_META = 8, /* library metadata (row offsets, lengths, flags)    */
    KVD_BUF_COUNT = 9
};

/* Layer descriptor.  Caller-allocated (host memory, plain bytes), filled by
 * kvd_layer_init and then owned by the library until the caller frees it;
 * its contents are private.  It mirrors on the host every length the
 * kernels need, so no call reads device memory back. */
typedef struct kvd_layer {
    uint64_t opaque[128];
} kvd_layer;

/* Sizes of a layer's buffers (cortiq LayerKvCache: one contiguous region
 * per live KV head per sequence, rows of head_dim values).
 *   n_seq      sequences in the batch (each is its own conversation);
 *   n_kv       KV heads; head_dim 64 or 128;
 *   mode       kvd_mode;
 *   capacity   host [n_seq], the most rows each sequence may ever hold
 *              (rounded up to a multiple of 16 internally);
 *   alive      host [n_kv], 0 = dead KV head (stores nothing, its query
 *              heads produce zeros), NULL = all alive;
 *   bytes_out  host [KVD_BUF_COUNT] device bytes per slot (0 = unused);
 *   host_bytes_out  bytes of the host state block kvd_layer_init needs.
 * Layout of every row buffer: sequence-major, then live head, then row:
 * [seq][live head][row][...], sequence b occupying n_live * cap_b rows. */
KVD_API kvd_status kvd_layer_bytes(int32_t n_seq, int32_t n_kv, int32_t head_dim, int32_t mode,
                           const int64_t *capacity, const uint8_t *alive,
                           int64_t *bytes_out, int64_t *host_bytes_out);

/* Bind L to caller buffers (device pointers in dev_bufs[KVD_BUF_COUNT],
 * each 256-byte aligned, sized by kvd_layer_bytes; host_state of
 * host_bytes_out bytes) and clear every sequence: length 0, fields unset
 * (stored as 1.0).  Enqueues the metadata upload and field reset on
 * `stream`; host_state must stay alive and unmoved while L is in use. */
KVD_API kvd_status kvd_layer_init(kvd_layer *L, int32_t n_seq, int32_t n_kv, int32_t head_dim,
                          int32_t mode, const int64_t *capacity, const uint8_t *alive,
                          void *const *dev_bufs, void *host_state, void *stream);

/* cortiq clear: forget sequence `seq` (or every sequence, seq = -1): length
 * 0, fields unset.  Row contents are left in place and never read again. */
KVD_API kvd_status kvd_layer_reset(kvd_layer *L, int32_t seq, void *stream);

/* Host-mirrored state: rows stored by sequence `seq`, and whether its
 * channel fields are frozen.  Synchronous, reads no device memory. */
KVD_API kvd_status kvd_layer_seq_len(const kvd_layer *L, int32_t seq, int64_t *len_out,
                             int32_t *frozen_out);

/* cortiq memory_bytes summed over the batch: f32 rows, scales and frozen
 * fields at 4 bytes, int8 codes at 1 byte, for the rows currently stored. */
KVD_API kvd_status kvd_layer_memory_bytes(const kvd_layer *L, int64_t *bytes_out);

/* cortiq LayerKvCache::append (+ quant_row), batched over sequences.
 *   k, v   device f32 [sum n_new][n_kv][head_dim]: the new rows of sequence
 *          0, then of sequence 1, ...; dead heads' slices are ignored;
 *   n_new  host [n_seq] rows appended per sequence, or NULL for one row
 *          each (k, v then hold [n_seq][n_kv][head_dim]).
 * Each row of a quantised component is divided by its channel field (1
 * before the freeze) and coded per group: scale = max(absmax/127, 1e-12),
 * code = clamp(round_half_even(r / scale), -127, 127), f32 IEEE throughout.
 * Semantics are those of appending the rows one at a time: the freeze of
 * kv_freeze_colfield runs before the first row appended while the sequence
 * holds >= 64 rows with its fields unset.  KVD_ECAPACITY if any sequence
 * would exceed its capacity (nothing is appended then). */
KVD_API kvd_status kv_append(kvd_layer *L, const float *k, const float *v, const int32_t *n_new,
                     void *stream);

/* cortiq freeze_cols for every sequence that holds >= 64 rows and has no
 * field yet (a no-op for the others and for KVD_F32): per live head and
 * quantised component, dequantise the stored rows, col[d] = max(sqrt(
 * sum_p row[p][d]^2 / n), 1e-6) in row order with IEEE rounding of every
 * operation, then requantise every stored row against col.  Idempotent. */
KVD_API kvd_status kv_freeze_colfield(kvd_layer *L, void *stream);

/* Workspace bytes decode_attention_verify needs for n_q query heads and K drafts. */
KVD_API kvd_status kvd_verify_workspace_bytes(const kvd_layer *L, int32_t n_q, int32_t K,
                                              int64_t *bytes_out);

/* Query-batched verify of K draft rows (speculative decode), read as cortiq
 * attend_group_upto's causal limit: the K drafts have been appended
 * (kv_append), so sequence b holds L_b rows ending with them; query k
 * (q device f32 [n_seq][K][n_q][head_dim]) attends rows [first_k, upto_k)
 * with upto_k = L_b - (K - 1 - k) -- everything before draft k and draft k
 * itself, causal among the drafts -- first_k = upto_k - window when
 * upto_k > window (else 0), softcap and sinks as decode_attention_ex.  Every
 * K/V row is read once for the K * n_q queries (n_q / n_kv * K <= 16).
 * out device f32 [n_seq][K][n_q][head_dim]; a query whose upto_k <= 0 gets
 * zeros.  No imp (rejected drafts are dropped by kv_truncate_last).  With
 * K = 1 it is decode_attention_ex without imp. */
KVD_API kvd_status decode_attention_verify(const float *q, const kvd_layer *L, int32_t n_q, int32_t K,
                                           float scale, int64_t window, float softcap,
                                           const float *sinks, float *out, void *workspace,
                                           int64_t workspace_bytes, void *stream);

/* cortiq LayerKvCache::truncate_last (speculative-decode reject), batched:
 * sequence b drops its last min(n_drop[b], length) rows in every storage
 * (n_drop host [n_seq], NULL = one row each).  Only the lengths change;
 * with imp (device f32, the decode_attention buffer, or NULL) the dropped
 * rows' entries are cleared so that rows appended later start from zero
 * mass.  Frozen fields are kept.  KVD_EINVAL for a negative count. */
KVD_API kvd_status kv_truncate_last(kvd_layer *L, const int32_t *n_drop, float *imp, void *stream);

/* Workspace bytes kv_evict_born needs for a given keep_last: the kept-row
 * lists and a copy of their masses (keep_last entries each for up to 256
 * sequences), the select's per-sequence state, digit histograms and
 * per-4096-row chunk counts, plus, for layers with few (sequence, live head,
 * storage) regions, up to 64 MiB of staging for the batched gather.  No
 * initialisation needed. */
KVD_API kvd_status kv_evict_workspace_bytes(const kvd_layer *L, int64_t keep_last, int64_t *bytes_out);

/* cortiq LayerKvCache::evict_born for every sequence of the layer holding
 * more than keep_last rows (the others are left alone): keep its first
 * min(sink, keep_last) rows (attention sinks), its last min(recent,
 * keep_last - sinks) rows, and fill the rest of the keep_last budget with
 * the middle rows of highest accumulated mass imp (equal mass: the lower
 * row first); the kept rows move, in row order, to rows 0 .. keep_last - 1
 * of every storage of every live head independently (f32 K / V, int8 codes
 * and their scales), imp moves with them (the dropped rows' entries are
 * cleared, so rows appended later start from zero mass), and the sequence's
 * length becomes keep_last.  Frozen fields are kept.  cortiq KvCache::evict under
 * EvictionPolicy::Born { sink } passes recent = max(keep_last / 2, 1).
 *   imp        device f32, the buffer decode_attention accumulates
 *              (imp_off(b) + p); masses must be finite;
 *   workspace  device, 256-byte aligned, >= kv_evict_workspace_bytes.
 * KVD_EINVAL for a negative keep_last, sink or recent. */
KVD_API kvd_status kv_evict_born(kvd_layer *L, float *imp, int64_t keep_last, int32_t sink,
                                 int32_t recent, void *workspace, int64_t workspace_bytes,
                                 void *stream);

/* Workspace bytes decode_attention needs for n_q query heads (with_imp != 0
 * adds the score buffer the imp pass uses).  Depends only on the layer's
 * shape and capacities, so one allocation serves every later call. */
KVD_API kvd_status kvd_decode_workspace_bytes(const kvd_layer *L, int32_t n_q, int32_t with_imp,
                                      int64_t *bytes_out);

/* Single-token GQA decode attention over the layer (cortiq attend_group
 * over every KV group): query head h reads KV head h / (n_q / n_kv);
 *   out[b][h] = sum_p softmax_p(scale * <q[b][h], K^[p]>) V^[p]
 * over the rows stored for sequence b, with K^ = code * scale * kcol, V^ =
 * code * scale * vcol for quantised components.  Split over the SMs by
 * position chunks (flash-decoding) and merged by log-sum-exp.
 *   q    device f32 [n_seq][n_q][head_dim];  out device f32, same shape;
 *   imp  device f32 or NULL: imp[imp_off(b) + p] += sum over live query
 *        heads of their softmax weight on row p (cortiq accumulate_imp);
 *        imp_off(b) = sum of the (16-rounded) capacities of the sequences
 *        before b, so imp holds sum_b cap_b floats;
 *   workspace  device, >= kvd_decode_workspace_bytes(L, n_q, imp != NULL).
 * Dead groups and empty sequences give zeros and leave imp unchanged.
 * n_q must be a multiple of n_kv with n_q / n_kv <= 16. */
KVD_API kvd_status decode_attention(const float *q, const kvd_layer *L, int32_t n_q, float scale,
                            float *out, float *imp, void *workspace, int64_t workspace_bytes,
                            void *stream);

/* decode_attention with the options of cortiq attend_group_upto (docs.rs
 * cortiq-engine 0.8.49, kv_cache.rs, attend_group / attend_group_upto):
 *   window   >= 0; 0 = every stored row.  Otherwise sequence b (L_b rows)
 *            sees rows [first_b, L_b) with first_b = L_b - window when L_b >
 *            window, else 0 -- the page's `first` as sliding-window layers
 *            pass it; earlier rows get probability 0 and their imp entries
 *            are left unchanged;
 *   softcap  >= 0, finite; > 0 replaces every computed score s = scale *
 *            <q, K^> by softcap * tanh(s / softcap) before the softmax
 *            (logit soft-capping; the sink is not capped);
 *   sinks    device f32 [n_q] or NULL: a learned sink logit per query head
 *            that joins the softmax maximum and adds exp(sink - max) to its
 *            denominator, with no value row (so the rows' weights, out and
 *            imp shrink by the sink's share).
 * Every other argument, the workspace size and the errors are those of
 * decode_attention, which is this call with window 0, softcap 0 and no
 * sinks.  Returns KVD_EINVAL for a negative window, a negative or
 * non-finite softcap, or a misaligned sinks pointer. */
KVD_API kvd_status decode_attention_ex(const float *q, const kvd_layer *L, int32_t n_q, float scale,
                               int64_t window, float softcap, const float *sinks, float *out,
                               float *imp, void *workspace, int64_t workspace_bytes, void *stream);

/* decode_attention for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a deployment variant).  Some callers cannot
 * call cudaMalloc on their decode path -- an inference runtime that hands out
 * device memory from a fixed, pre-planned arena, a plug-in inside a host
 * application that owns every allocation, code that must not take
 * cudaMalloc's implicit device-wide synchronisation while serving -- so this
 * call takes no workspace: its scratch (the per-chunk partial results) lives
 * in a 16 MiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits.  It allocates nothing and computes
 * the same outputs as decode_attention with imp = NULL.
 *   Limit: n_seq * n_live * chunks * (n_q / n_kv) * (2 + head_dim) * 4 bytes
 *   (each region rounded up to 256) must fit in 16 MiB, where chunks is the
 *   longest sequence divided by the rows per chunk the call picks (>= 256);
 *   a larger call returns KVD_ECAPACITY and launches nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and keeps it with the id of the current context; a
 *   call under another context (after a device reset, which unloads the
 *   module and the array with it) looks it up again.  Make the first call on
 *   a device, and the first after a reset, before any stream capture.  Calls
 *   share the array and it keeps the last call's partials: two calls whose
 *   kernels overlap on the GPU race and must be serialised by the caller. */
KVD_API kvd_status decode_attention_static(const float *q, const kvd_layer *L, int32_t n_q,
                                           float scale, float *out, void *stream);

/* Device error word of the layer (0 = clean), copied back synchronously;
 * clear != 0 resets it.  Bit 0: a bounded wait timed out; bit 1: a kernel
 * found metadata out of range and skipped the access. */
KVD_API kvd_status kvd_layer_device_error(const kvd_layer *L, int32_t clear, uint32_t *word_out);

/* Failure injection for tests (the pages have no counterpart; host-only, the
 * device never sees it).  n >= 0 arms a process-wide counter: the (n+1)-th
 * kernel launch or host/device copy that the library issues from then on
 * reports failure, the entry point that issued it returns KVD_ECUDA, and the
 * counter disarms itself; n < 0 disarms it.  Entry points that change
 * host-mirrored state (lengths, frozen flags, ring cursors, histories) change
 * it only after every launch of the call has gone in, so a call that fails
 * this way leaves that state as it was; kernels it launched before the
 * failure may have run, so the caller resets the layer or stream state it
 * cannot vouch for (kvd_layer_reset).  Calls from several threads at once
 * share the counter. */
KVD_API kvd_status kvd_test_fail_after(int64_t n);

/* The bounded-wait path, run on purpose (a diagnostic: the pages have no
 * counterpart).  One warp waits for an mbarrier phase that nothing
 * completes, gives up after limit_ns nanoseconds and sets bit 0 of the
 * layer's device error word, as a decode kernel whose copies never landed
 * would; the kernel exits normally and the context stays usable.  Read the
 * word with kvd_layer_device_error after synchronising the stream.
 * KVD_EINVAL for limit_ns outside 1 .. 10^9. */
KVD_API kvd_status kvd_wait_timeout_selftest(const kvd_layer *L, int64_t limit_ns, void *stream);

/* The kernels' metadata guards, run on purpose (a diagnostic: the pages have
 * no counterpart; it exercises bit 1 of the device error word, which no
 * sequence of ordinary calls sets).  Launches, on `stream`: the append kernel
 * asked for storage row cap[0] of sequence 0 (one past its capacity); for a
 * quantised mode the freeze kernel on lengths that put sequence 0 at
 * cap[0] + 1 rows; and the decode's split kernel on the same lengths (one CTA
 * on the CUDA-core path, one worker over one tile on the q8_2f tensor-core
 * path).  The fake lengths, and every length, flag, partial or slot record
 * those kernels are given to write, live in `scratch` (device, caller-owned,
 * 256-byte aligned, at least kvd_bounds_selftest_bytes bytes; its contents on
 * return are unspecified), never in the layer.  Each kernel's guard sets
 * bit 1 and returns before it reads or writes the cache, so the layer's
 * storage, lengths and frozen flags are unchanged.  Read the word with
 * kvd_layer_device_error after synchronising the stream.  KVD_EINVAL for a
 * layer without live groups, a null or unaligned scratch, or cap[0] >= 2^31 - 1;
 * KVD_ECAPACITY if scratch_bytes is too small (nothing launched). */
KVD_API kvd_status kvd_bounds_selftest_bytes(const kvd_layer *L, int64_t *bytes_out);
KVD_API kvd_status kvd_bounds_selftest(const kvd_layer *L, void *scratch, int64_t scratch_bytes, void *stream);

/* ---- R-SWA (rswa module): retained prefix + W-slot ring, per stream ----
 * Per stream s and head h the reference block is ref[s][h][0..ref_cap) and
 * the ring ring[s][h][0..W), rows of head_dim f32 (head-major, as rswa
 * RingCache keeps them).  Cursors live on the host, one int32 per stream:
 * prefill_len (< 0 = no prefill recorded), ring_len, ring_pos.  The
 * writers also keep, when given a host rswa_history array [B], each
 * stream's decode-write count and branch lineage (rswa RingCache's
 * decode_writes and lineage_epoch), which rswa_checkpoint_take and
 * rswa_rollback_to use; NULL = not kept. */
typedef struct {
    int64_t decode_writes;   /* ring writes since the stream's prefill */
    uint64_t lineage_epoch;  /* +1 at every prefill and every rollback that discards writes */
} rswa_history;

/* rswa RingCache::record_prefill for stream `s`: copy k, v (device f32
 * [H][seq][head_dim]) into the reference block and reset the stream's ring
 * (ring_len = ring_pos = 0; with hist: decode_writes = 0 and a new
 * lineage).  KVD_ECAPACITY if seq > ref_cap; KVD_ESTATE if the lineage
 * counter is exhausted. */
KVD_API kvd_status rswa_record_prefill(float *ref_k, float *ref_v, const float *k, const float *v,
                               int32_t s, int32_t seq, int32_t B, int32_t H, int32_t head_dim,
                               int64_t ref_cap, int32_t W, int32_t *prefill_len,
                               int32_t *ring_len, int32_t *ring_pos, rswa_history *hist,
                               void *stream);

/* rswa RingCache::write_decode_step for every stream at once: stream s
 * writes its token (k, v device f32 [B][H][head_dim], already rotated at
 * the true absolute position by the caller) into slot ring_len[s] while
 * ring_len < W (then ring_len += 1, ring_pos = ring_len % W) and into slot
 * ring_pos[s] afterwards (then ring_pos = (ring_pos + 1) % W).  Cursors are
 * host arrays updated in place (with hist: decode_writes += 1); slot_out
 * (host [B] or NULL) gets each stream's slot.  KVD_ESTATE if any stream
 * has no prefill (nothing written). */
KVD_API kvd_status rswa_ring_write(float *ring_k, float *ring_v, const float *k, const float *v,
                           const int32_t *prefill_len, int32_t *ring_len, int32_t *ring_pos,
                           rswa_history *hist, int32_t B, int32_t H, int32_t head_dim, int32_t W,
                           int32_t *slot_out, void *stream);

/* rswa RingCheckpoint of one stream: the issuing cache's identity (a
 * caller-chosen number), the prefill boundary, the ring cursors, the
 * decode-write count and the lineage at the time it was taken. */
typedef struct {
    uint64_t cache_id;
    uint64_t lineage_epoch;
    int64_t decode_writes;
    int32_t prefill_len, ring_len, ring_pos, pad;
} rswa_checkpoint;

/* rswa RingCache::checkpoint of stream s (host only, O(1), no K/V copy). */
KVD_API kvd_status rswa_checkpoint_take(uint64_t cache_id, const int32_t *prefill_len,
                                        const int32_t *ring_len, const int32_t *ring_pos,
                                        const rswa_history *hist, int32_t s, rswa_checkpoint *out);

/* rswa RingCache::rollback_to for stream s (host only): restore ring_len,
 * ring_pos and decode_writes from cp, discarding the ring writes made since
 * (the stale slots >= ring_len are never read).  Refused with KVD_ESTATE,
 * nothing changed, when cp comes from another cache, another prefill
 * boundary or another lineage, is from the future, or when the discarded
 * writes wrapped the ring over a row live at the checkpoint (cp.ring_len +
 * discarded > W: an overwritten row cannot be restored from cursors).  A
 * rollback that discards writes starts a new lineage. */
KVD_API kvd_status rswa_rollback_to(uint64_t cache_id, const int32_t *prefill_len, int32_t *ring_len,
                                    int32_t *ring_pos, rswa_history *hist, int32_t s, int32_t W,
                                    const rswa_checkpoint *cp);

/* Workspace bytes rswa_decode needs. */
KVD_API kvd_status rswa_decode_workspace_bytes(int32_t B, int32_t H, int32_t head_dim,
                                       int64_t ref_cap, int32_t W, int64_t *bytes_out);

/* rswa decode_attention for every stream: per (stream, head) softmax over
 * reference rows [0, prefill_len) followed by ring rows [0, ring_len),
 * no mask, scale `scale`; out device f32 [B][H * head_dim].  ring_pos is
 * accepted for the cursor contract only (attention over the ring does not
 * depend on the order of its slots).  KVD_ESTATE if a stream has no
 * prefill, KVD_EEMPTY if one has no keys.  ws >= rswa_decode_workspace_bytes;
 * its first 4 bytes are the device error word (rswa_device_error), which the
 * caller zeroes once before the first call. */
KVD_API kvd_status rswa_decode(const float *q, const float *ref_k, const float *ref_v,
                       const float *ring_k, const float *ring_v, const int32_t *prefill_len,
                       const int32_t *ring_len, const int32_t *ring_pos, int32_t B, int32_t H,
                       int32_t head_dim, int64_t ref_cap, int32_t W, float scale, float *out,
                       void *workspace, int64_t workspace_bytes, void *stream);

/* ---- R-SWA int8 mirror (rswa Int8Kv, quantize_row_i8,
 * decode_attention_int8) ----
 * A per-row symmetric int8 copy of the four f32 regions, kept beside them
 * (the f32 regions stay the source of truth).  Codes have the regions'
 * shapes, [B][H][ref_cap][head_dim] and [B][H][W][head_dim]; each row has
 * one f32 scale, [B][H][ref_cap] and [B][H][W].  A row's scale is
 * max|x| / 127 (1.0 for an all-zero row) and its codes are
 * clamp(round_half_even(x / scale), -127, 127), IEEE f32 division.  All
 * eight are device pointers owned by the caller, 16-byte aligned. */
typedef struct {
    int8_t *ref_k, *ref_v;
    float *ref_ks, *ref_vs;
    int8_t *ring_k, *ring_v;
    float *ring_ks, *ring_vs;
} rswa_i8_mirror;

/* rswa_record_prefill plus the int8 mirror of the copied rows (rswa
 * RingCache::record_prefill with the int8 lever on: the whole reference block
 * is mirrored once).  head_dim 64 or 128; k, v, ref_k, ref_v 16-byte aligned.
 * Same cursor update and errors as rswa_record_prefill. */
KVD_API kvd_status rswa_record_prefill_i8(float *ref_k, float *ref_v, const rswa_i8_mirror *m,
                                          const float *k, const float *v, int32_t s, int32_t seq,
                                          int32_t B, int32_t H, int32_t head_dim, int64_t ref_cap,
                                          int32_t W, int32_t *prefill_len, int32_t *ring_len,
                                          int32_t *ring_pos, rswa_history *hist, void *stream);

/* rswa_ring_write plus the int8 mirror of each freshly written ring row at the
 * same slot (rswa write_decode_step with the int8 lever on).  head_dim 64 or
 * 128; k, v, ring_k, ring_v 16-byte aligned.  Same cursor update, slot_out
 * and errors as rswa_ring_write. */
KVD_API kvd_status rswa_ring_write_i8(float *ring_k, float *ring_v, const rswa_i8_mirror *m,
                                      const float *k, const float *v, const int32_t *prefill_len,
                                      int32_t *ring_len, int32_t *ring_pos, rswa_history *hist,
                                      int32_t B, int32_t H, int32_t head_dim, int32_t W,
                                      int32_t *slot_out, void *stream);

/* rswa decode_attention_int8 for every stream, reading the int8 mirror only:
 * per (stream, head) the query row is quantised like a cache row (codes and
 * qscale); each key's score is the exact integer dot of the codes times
 * qscale times the key row's K scale times `scale`; softmax over reference
 * rows [0, prefill_len) followed by ring rows [0, ring_len); V rows are
 * dequantised per row (code times the row's V scale).  out device f32
 * [B][H * head_dim].  Same cursor contract, workspace
 * (rswa_decode_workspace_bytes), alignment rules and errors as rswa_decode. */
KVD_API kvd_status rswa_decode_i8(const float *q, const rswa_i8_mirror *m,
                                  const int32_t *prefill_len, const int32_t *ring_len,
                                  const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                                  int64_t ref_cap, int32_t W, float scale, float *out,
                                  void *workspace, int64_t workspace_bytes, void *stream);

/* Workspace bytes rswa_verify / rswa_verify_i8 need for K drafts. */
KVD_API kvd_status rswa_verify_workspace_bytes(int32_t B, int32_t H, int32_t head_dim, int64_t ref_cap,
                                               int32_t W, int32_t K, int64_t *bytes_out);

/* rswa verify_attention for every stream, query-batched: K draft tokens
 * (q, draft_k, draft_v device f32 [B][K][H][head_dim], already rotated) are
 * attended as K sequential write_decode_step + decode_attention calls would
 * -- query i sees the reference rows and the last W rows of (the live ring
 * in logical order, then drafts 0..i): drafts that a full ring makes evict
 * its oldest rows -- WITHOUT writing the cache (it is read-only here; the
 * caller then writes the accepted drafts with rswa_ring_write).  The
 * reference rows are read once for all K queries of a head.  out device f32
 * [B][K][H * head_dim].  1 <= K <= 16; errors as rswa_decode (KVD_ESTATE for
 * a stream without prefill). */
KVD_API kvd_status rswa_verify(const float *q, const float *draft_k, const float *draft_v, int32_t K,
                               const float *ref_k, const float *ref_v, const float *ring_k,
                               const float *ring_v, const int32_t *prefill_len, const int32_t *ring_len,
                               const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                               int64_t ref_cap, int32_t W, float scale, float *out, void *workspace,
                               int64_t workspace_bytes, void *stream);

/* rswa_verify over the int8 mirror (decode_attention_int8): the drafts are
 * quantised per row as write_decode_step would mirror them, and each draft
 * query as decode_attention_int8 quantises a query.  At head_dim 128 with
 * K <= 8, ref_cap a multiple of 32 and B * H * ref_cap < 2^31 the reference
 * rows are read by the tensor-core kernel (TMA over the mirror's codes: their
 * base pointers must then also suit a TMA descriptor, which the 16-byte rule
 * above does; if the driver refuses one, the CUDA-core kernel runs); otherwise
 * by the CUDA-core kernel.  Same results within the output tolerance either
 * way; same workspace (rswa_verify_workspace_bytes covers both). */
KVD_API kvd_status rswa_verify_i8(const float *q, const float *draft_k, const float *draft_v, int32_t K,
                                  const rswa_i8_mirror *m, const int32_t *prefill_len,
                                  const int32_t *ring_len, const int32_t *ring_pos, int32_t B, int32_t H,
                                  int32_t head_dim, int64_t ref_cap, int32_t W, float scale, float *out,
                                  void *workspace, int64_t workspace_bytes, void *stream);

/* Device error word kept in an R-SWA workspace (see kvd_layer_device_error). */
KVD_API kvd_status rswa_device_error(const void *workspace, int32_t clear, uint32_t *word_out);

/* Short English description of a status code (static storage). */
KVD_API const char *kvd_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* KVD_H */
