/*
 * kvc.h -- grouped-query attention over a contiguous preallocated KV cache.
 *
 * C ABI of libkvc.so (GB300 / sm_103a).  Plain pointers and sizes only.
 *
 * The operation (three web pages, cited by title and section):
 *  - "Implement grouped-query attention over a preallocated KV cache, with no
 *    torch.cat, for both prefill chunks and decode" (inferenceinterviews.com),
 *    section "A strong answer": K and V are allocated once as
 *    [B, Hkv, max_len, d]; a call writes the new chunk in place at each row's
 *    current length (KVCache.append) and then lets the chunk's T queries
 *    attend (gqa_attention) with query head h reading KV head h / G
 *    (G = Hq / Hkv), scores scaled by 1/sqrt(d), query t of row b at absolute
 *    position lens[b] - n_new[b] + t, keys past lens[b] and padded queries
 *    (t >= n_new[b]) masked, and fully masked queries returning zeros.
 *  - "Write the causal mask for a decode step with a KV cache, where the query
 *    is shorter than the keys" (inferenceinterviews.com), TL;DR and "A strong
 *    answer": the mask is bottom-right aligned (key j visible to query i iff
 *    j <= i + S - T) and lives in the kernel as index arithmetic.
 *  - "16. Prefill, decode and the KV cache" (inference.shantanugoel.com),
 *    "Layout and validity": one K/V buffer pair per layer, per-layer lengths,
 *    a length query that refuses when layers disagree, truncate and reset.
 *
 * Layout.  Every tensor is dense, row-major, in the cache's element type
 * (KVC_F32 = float, KVC_BF16 = bfloat16):
 *   K, V cache of one layer   [B, Hkv, max_len, d]
 *   k_new, v_new              [B, Hkv, T, d]
 *   q, out                    [B, Hq, T, d]
 * All device pointers must be 16-byte aligned.  d * sizeof(element) must be a
 * multiple of 16, and d <= 256.  bf16 and FP8 caches of d = 128 run on the
 * TMA / tensor-core kernels.  fp32 caches, and bf16 or FP8 caches of any
 * other d, run on a generic kernel.  That kernel widens the stored values to
 * fp32 (an FP8 code times its head's scale).  It has no fused append, no device-resident steps
 * and no allocation-free entry point, and needs a workspace only for calls
 * whose key ranges it splits (kvc_workspace_bytes).
 *
 * Device.  One process drives one GPU through this library: a handle binds
 * to the device current at its first launching call, every later launching
 * call must find that device current, and handles of a second device in the
 * same process are refused (KVC_ERR_ARG).  Run one process per GPU.
 *
 * Threads.  A handle holds host state (lengths, descriptors) without a lock:
 * calls on one handle must not overlap in time.  Different handles may be
 * used from different threads.
 *
 * Ownership.  The caller allocates every device buffer (cache, inputs,
 * outputs, workspace) and keeps it alive while the handle or a launched call
 * uses it.  The handle owns only host state: per-layer, per-row lengths and
 * launch descriptors.  kvc_destroy frees the handle, never a buffer.
 *
 * Lengths are host-authoritative.  kvc_append grows lens only after its
 * kernel was enqueued successfully.  Kernels run asynchronously on the given
 * stream (a cudaStream_t passed as void*, NULL = legacy default stream).
 *
 * Errors.  Every entry point returns a kvc_status and never throws.  All
 * arguments are validated before anything is enqueued, so an error leaves
 * cache data, lengths and outputs untouched (the pages' "appending past
 * max_len raises and leaves the row's length unchanged", applied to every
 * row).  kvc_last_error() gives a message for the calling thread's last
 * failure.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of the cache.  q, out, k_new and v_new have the same type,
 * except for KVC_FP8_E4M3 caches: those store one byte per value (E4M3:
 * 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest finite 448,
 * no infinity) with one scale per (layer, KV head) for K and for V
 * (kvc_set_kv_scales), and take bf16 q / k_new / v_new / out ("16. Prefill,
 * decode and the KV cache", exercise 4: store the cache in FP8 E4M3 with one
 * scale per head and dequantize on read).  Their MMAs run in f16 (E4M3 and
 * bf16 convert to f16 exactly within f16's range), so an FP8 cache needs
 * |q| < 65504. */
typedef enum { KVC_F32 = 0, KVC_BF16 = 1, KVC_FP8_E4M3 = 2 } kvc_dtype;

typedef enum {
    KVC_OK = 0,
    KVC_ERR_ARG = 1,             /* bad pointer, size, dtype, alignment, layer index */
    KVC_ERR_SHAPE = 2,           /* Hq not a multiple of Hkv, n_new outside 0..T, ... */
    KVC_ERR_OVERFLOW = 3,        /* lens[b] + n_new[b] > max_len for some row */
    KVC_ERR_LAYER_MISMATCH = 4,  /* layers disagree on a row's length */
    KVC_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed (no GPU, launch error) */
    KVC_ERR_DEVICE_TIMEOUT = 6,  /* a kernel's bounded wait ran out (see kvc_device_status) */
    KVC_ERR_WORKSPACE = 7        /* workspace missing, too small or misaligned */
} kvc_status;

/* Largest batch the attention kernels accept (per-row offsets travel as
 * kernel parameters, so no device metadata buffer is needed). */
#define KVC_MAX_BATCH 1024

typedef struct kvc_cache kvc_cache;

/* Create a handle over caller-owned cache buffers.
 * k_bufs[l], v_bufs[l] (l < layers) each point to [B, Hkv, max_len, d]
 * elements of `dtype` on the current device.  All lengths start at 0.
 * No CUDA call is made here; device state (tensor-map descriptors, SM
 * count) is set up on the first launch.
 * Errors: KVC_ERR_ARG for non-positive sizes, B > KVC_MAX_BATCH, null or
 * misaligned buffers, d * element size not a multiple of 16, or d > 256;
 * FP8 caches take at most 64 KV heads. */
kvc_status kvc_create(kvc_cache** out, int layers, int batch, int kv_heads, int max_len, int head_dim,
                      kvc_dtype dtype, void* const* k_bufs, void* const* v_bufs);

/* Free the handle (not the cache buffers).  A handle that has served
 * kvc_append_attention_host first waits for its copies to finish, then frees
 * its device staging, copy streams and events.  NULL is accepted. */
void kvc_destroy(kvc_cache* c);

/* Scales of an FP8 E4M3 cache's layer: k_scale[h], v_scale[h] (host arrays of
 * kv_heads floats, copied) for KV head h.  Appends store a value x of head h
 * as the E4M3 code nearest to x * (1/s) (the reciprocal and the product each
 * rounded to float32; ties to even; beyond +-448 saturating to +-448), and
 * attention reads code * s.  Every scale starts at 1.  Only while every row
 * of the layer has length 0 (the stored codes depend on the scale).
 * Errors: KVC_ERR_ARG (not an FP8 cache, bad layer, null arrays, a scale not
 * positive and finite, or the layer holds data); nothing changes on error. */
kvc_status kvc_set_kv_scales(kvc_cache* c, int layer, const float* k_scale, const float* v_scale);

/* A cache whose K/V live in pages ("Implement grouped-query attention over a
 * preallocated KV cache...", "A strong answer", the reversal condition: rows of
 * wildly different lengths call for a block table; "16. Prefill, decode and the
 * KV cache", "Design choices worth noticing": a paged cache reserves no
 * max_len per row).  k_bufs[l] / v_bufs[l] are caller-owned device buffers
 * [num_pages, kv_heads, page_size, head_dim]; block_table is a caller-owned
 * device int32 [batch, max_pages_per_row]: row b's tokens
 * i * page_size .. (i + 1) * page_size - 1 live in page block_table[b][i]
 * (-1: not mapped).  Every later call works on the logical sequence exactly as
 * with kvc_create, with max_len = max_pages_per_row * page_size.  The caller
 * keeps the entries under every position a call appends or attends to valid
 * (0 .. num_pages - 1) and may change the table between calls (stream-ordered).
 * A bad entry is never dereferenced: appended rows aimed at it are not
 * written, and reads take page 0 and set the workspace error word (the next
 * kvc_device_status reports it); the generic kernel (fp32; bf16, FP8 of
 * d != 128) reads it as zeros.  bf16 and FP8 caches of d = 128, and bf16 caches of d = 64, need
 * page_size % 128 == 0 (a key tile lies in one page).  Paged storage does not combine with ring
 * storage (kvc_set_window ring = 1).  Errors: as kvc_create, and KVC_ERR_ARG
 * for bad paging arguments. */
kvc_status kvc_create_paged(kvc_cache** out, int layers, int batch, int kv_heads, int page_size, int num_pages,
                            int max_pages_per_row, int head_dim, kvc_dtype dtype, void* const* k_bufs,
                            void* const* v_bufs, const int32_t* block_table);

/* Append in place ("A strong answer", KVCache.append): for every row b and
 * t < n_new[b], copy k_new[b, :, t, :] to K[b, :, lens[b] + t, :] (same for
 * V), then lens[layer][b] += n_new[b].  n_new is a HOST array of B entries.
 * The copy is bit-exact.  Rows with n_new[b] = 0 are untouched.
 * Errors (nothing written, lens unchanged): KVC_ERR_ARG (layer, pointers,
 * T < 0), KVC_ERR_SHAPE (n_new[b] < 0 or > T), KVC_ERR_OVERFLOW
 * (lens[b] + n_new[b] > max_len for any row), KVC_ERR_CUDA (launch failed). */
kvc_status kvc_append(kvc_cache* c, int layer, const void* k_new, const void* v_new, int T,
                      const int32_t* n_new, void* stream);

/* Bytes of device workspace kvc_gqa_attention needs for this handle, q_heads
 * and T (an error word and the split-KV partial results).
 * 0 means no workspace is needed: the generic kernel (fp32 caches; bf16 and
 * FP8 caches of d != 128) needs one only for calls with few (row, KV head,
 * 16-row block) units, whose key ranges it splits across CTAs.  Returns 0 for invalid
 * input. */
size_t kvc_workspace_bytes(const kvc_cache* c, int q_heads, int T);

/* Attention of the chunk just appended ("A strong answer", gqa_attention):
 * q [B, Hq, T, d] -> out [B, Hq, T, d].  For t < n_new[b], out[b,h,t,:] is
 * the softmax(q.K^T / sqrt(d)) weighted sum of V over keys
 * 0 .. lens[b] - n_new[b] + t of KV head h / (Hq / Hkv); for t >= n_new[b]
 * it is 0.  lens are the current lengths of `layer` (after the append).
 * Accumulation is fp32; out has the cache's element type.
 * workspace: device buffer of at least kvc_workspace_bytes(c, Hq, T) bytes,
 * 256-byte aligned, used by one call at a time (calls that share a workspace
 * must be ordered on one stream).  Its contents need no initialisation: the
 * library clears the error word itself the first time a handle sees a
 * workspace pointer.
 * Errors (out untouched): KVC_ERR_ARG, KVC_ERR_SHAPE (Hq % Hkv != 0,
 * n_new[b] < 0, n_new[b] > T, n_new[b] > lens[b]), KVC_ERR_WORKSPACE,
 * KVC_ERR_CUDA. */
kvc_status kvc_gqa_attention(kvc_cache* c, int layer, const void* q, int q_heads, int T,
                             const int32_t* n_new, void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* kvc_append followed by kvc_gqa_attention with the same n_new, validated
 * together first: on any error neither step runs. */
kvc_status kvc_append_attention(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new,
                                int q_heads, int T, const int32_t* n_new, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Tree speculative verify ("Write the causal mask for a decode step with a KV
 * cache...", "What interviewers probe next": tree-based speculative
 * decoding).  The chunk's draft tokens form one tree per row, given by
 * parents (host int32 [B * T]): parents[b * T + t] in -1 .. t - 1 for
 * t < n_new[b] (a parent precedes its child; -1: the token hangs directly off
 * the cached prefix; entries for t >= n_new[b] are ignored).  Query t then
 * sees every key before the chunk plus the chunk's tokens on its own path to
 * the root (itself and its ancestors) instead of the triangle; everything
 * else is as in kvc_gqa_attention / kvc_append_attention.  Limits: T <= 64,
 * B * T <= 1024, no sliding window; bf16 caches take G * T <= 64 query rows
 * per KV head.  Errors (nothing enqueued): those of the plain calls, and
 * KVC_ERR_SHAPE for a parent outside -1 .. t-1 or a shape past the limits,
 * KVC_ERR_ARG for a null parents or a cache with a window. */
kvc_status kvc_gqa_attention_tree(kvc_cache* c, int layer, const void* q, int q_heads, int T,
                                  const int32_t* n_new, const int32_t* parents, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);
kvc_status kvc_append_attention_tree(kvc_cache* c, int layer, const void* q, const void* k_new,
                                     const void* v_new, int q_heads, int T, const int32_t* n_new,
                                     const int32_t* parents, void* out, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* kvc_append_attention with q, k_new, v_new and out in HOST memory (the same
 * shapes, [B, Hq, T, d] and [B, Hkv, T, d], element type as there: bf16 for an
 * FP8 cache), for a caller whose step inputs start and whose outputs end on the
 * host ("A strong answer": KVCache.append then gqa_attention, one decode or
 * prefill step).  Host buffers should be page-locked (cudaHostAlloc or
 * cudaHostRegister) so that the copies run asynchronously; all four must be
 * 16-byte aligned.
 * Only positions t < n_new[b] move: those of q, k_new and v_new to the device,
 * those of out back to out_host.  Positions t >= n_new[b] of out_host are not
 * written (kvc_append_attention would have written zeros there).
 * The call returns once it has enqueued: the input copies on a copy stream of
 * the handle, the append and attention on `stream`, the output copy on a
 * second copy stream.  Two device staging slots of the handle alternate from
 * call to call, so one call's output copy and the next call's input copies
 * overlap the compute in between.  The input buffers must stay unchanged, and
 * out_host unread, until kvc_host_copies_done has made a stream wait and that
 * stream has reached the wait (for example cudaStreamSynchronize after it).
 * The staging slots are allocated on the first call and grown, after the
 * calls that use them have finished, when a call needs more; kvc_destroy
 * frees them.  Each slot holds one call's q, k_new, v_new and out:
 * 2 * B * (Hq + Hkv) * T * d elements, each region rounded up to 256 bytes
 * (two slots: 84 MB for a bf16 chunk of B = 4, Hq = 32, Hkv = 8, T = 512,
 * d = 128).  Calls on one handle must come from one host thread in order.
 * Errors: those of kvc_append_attention, all found before anything is
 * enqueued or any host buffer is read (nothing is written, lengths
 * unchanged), and KVC_ERR_CUDA when a copy, an allocation or a launch fails. */
kvc_status kvc_append_attention_host(kvc_cache* c, int layer, const void* q_host, const void* k_host,
                                     const void* v_host, int q_heads, int T, const int32_t* n_new, void* out_host,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Make `stream` wait until every output copy of the host-buffer calls
 * enqueued so far on this handle has reached its host buffer (and so every
 * input copy before it).  Returns at once, without waiting on the host.
 * Errors: KVC_ERR_ARG (null handle), KVC_ERR_CUDA. */
kvc_status kvc_host_copies_done(kvc_cache* c, void* stream);

/* Size of the device scratch array behind kvc_gqa_attention_noalloc. */
#define KVC_NOALLOC_SCRATCH_BYTES (32u << 20)

/* kvc_gqa_attention without a workspace argument, for callers that cannot
 * allocate device memory: for instance a plugin inside a host program that
 * owns the whole device-memory budget and gives libraries no allocator, or
 * a latency-critical loop that must not pay cudaMalloc's cost and implicit
 * synchronization.  The pages have no counterpart of this entry point; it
 * computes exactly what kvc_gqa_attention computes (same kernel, same
 * result) and serves bf16 and FP8 caches of d = 128.
 *
 * Its scratch is one static device array of KVC_NOALLOC_SCRATCH_BYTES
 * (32 MiB) inside the library: every GPU that loads the library holds it
 * until the process exits.  No cudaMalloc, cudaFree or other allocating
 * call is made.  Calls with more than 12 query rows per KV head (G * T; 32
 * for FP8 caches) run on the tensor-core kernel, which needs only the workspace header and
 * uses the rest of the array for the partials of the items it cuts; they
 * always fit.  A call with fewer rows per KV head whose split-KV
 * scratch would exceed the array (very large batches; kvc_workspace_bytes
 * gives its size) is rejected with KVC_ERR_WORKSPACE before anything is
 * enqueued; decode shapes of batches up to 64 rows fit.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  The cached address belongs to the
 * device's current context: after cudaDeviceReset it is stale, like every
 * kvc handle and device buffer of that context, so a process that resets a
 * device must not call this entry point again.  Every call on a device
 * shares the one array, which keeps the last call's contents; each call
 * clears the part that must start at zero (the header's counters).  The
 * array's error word is not cleared by a call: a kernel's error (an expired
 * bounded wait, a bad block-table entry) stays recorded until
 * kvc_noalloc_status reads it.  Calls that overlap on the GPU (different
 * streams, or several caches at once) race on the array: order them on one
 * stream.  The device must be the cache's device (else KVC_ERR_ARG). */
kvc_status kvc_gqa_attention_noalloc(kvc_cache* c, int layer, const void* q, int q_heads, int T,
                                     const int32_t* n_new, void* out, void* stream);

/* kvc_device_status for the static scratch of kvc_gqa_attention_noalloc on
 * the current device: synchronizes `stream`, stores the scratch's error word
 * in *code (0 = every allocation-free call since the last read ran clean)
 * and clears it, and returns the same statuses as kvc_device_status
 * (KVC_ERR_DEVICE_TIMEOUT, KVC_ERR_OVERFLOW, or KVC_ERR_ARG for a block-table
 * entry outside 0 .. num_pages - 1).  Allocates nothing.  The pages have no
 * counterpart of this call. */
kvc_status kvc_noalloc_status(void* stream, int32_t* code);

/* Sliding window and ring storage ("Write the causal mask for a decode step
 * with a KV cache...", "A strong answer", last paragraph, and "Common
 * mistakes"; "16. Prefill, decode and the KV cache", exercise 3).
 *
 * window > 0: the query at absolute position p attends only to the keys at
 * positions a with p - window < a <= p (window = 0: all keys 0..p).
 * ring = 1: the cache is a ring of max_len slots per (row, KV head); the key
 * at position a lives in slot a mod max_len, and keys are chosen by position,
 * never by slot.  Lengths then count every token appended and may pass
 * max_len; each call's n_new[b] must be <= max_len - window + 1 (so the
 * chunk's first query still finds its window; else KVC_ERR_OVERFLOW), and
 * kvc_truncate may only go back to a length n whose window keys
 * n - window + 1 .. n - 1 are still stored (or to 0).
 * Requirements: ring needs 1 <= window <= max_len and, for bf16 and FP8
 * caches of d = 128 and bf16 caches of d = 64, max_len % 128 == 0 (a key
 * tile never wraps); ring storage changes only while every length is 0.
 * Applies to every layer and to every later call (including
 * kvc_decode_step).  Host only.  KVC_ERR_ARG otherwise. */
kvc_status kvc_set_window(kvc_cache* c, int window, int ring);

/* Forget everything after new_lens[b] tokens of row b in every layer
 * ("Layout and validity", truncate; speculative-decoding rollback).  No data
 * moves.  Requires the layers to agree (else KVC_ERR_LAYER_MISMATCH) and
 * 0 <= new_lens[b] <= length[b] (else KVC_ERR_ARG).  Host only. */
kvc_status kvc_truncate(kvc_cache* c, const int64_t* new_lens);

/* Set every length of every layer to 0 (truncate to 0).  Host only. */
kvc_status kvc_reset(kvc_cache* c);

/* Declare that the first lens[b] slots of every row of `layer` already hold
 * valid K/V (written by another producer or restored from storage), i.e.
 * set lens[layer][b] = lens[b].  Host only; no data moves.  Requires
 * 0 <= lens[b] <= max_len (else KVC_ERR_ARG, nothing changed).  This is the
 * one way to start from a non-empty cache without appending through it. */
kvc_status kvc_set_lens(kvc_cache* c, int layer, const int64_t* lens);

/* Copy lens[layer][0..B) into out (host array). */
kvc_status kvc_get_lens(const kvc_cache* c, int layer, int64_t* out);

/* Per-row length shared by all layers ("Layout and validity", length).
 * KVC_ERR_LAYER_MISMATCH if a forward pass stopped part-way (layers differ). */
kvc_status kvc_length(const kvc_cache* c, int64_t* out);

/* Read the device error word of a workspace used by handle c after the
 * stream's work ends: synchronizes `stream`, copies the word and stores it in
 * *code (0 = clean; otherwise a kernel's bounded wait expired and that call's
 * output is not valid), then clears the word.  Returns KVC_ERR_DEVICE_TIMEOUT
 * when *code != 0, KVC_ERR_OVERFLOW when the code records a rejected
 * device-resident step (kvc_decode_step), or KVC_ERR_ARG when a kernel met a
 * block-table entry outside 0 .. num_pages - 1 (kvc_create_paged; nothing was
 * read from or written to it, and that call's output is not valid).
 * A workspace that no call has used yet holds no status: its word is
 * whatever the buffer held (zero it, or make a call with it first). */
kvc_status kvc_device_status(kvc_cache* c, void* workspace, void* stream, int32_t* code);

/* Self-test of the kernels' bounded waits: launches one CTA that waits on an
 * mbarrier nothing ever arrives at, for at most limit_ns nanoseconds, then
 * writes its error code into the workspace's error word (the first 4 bytes),
 * so a following kvc_device_status reports KVC_ERR_DEVICE_TIMEOUT.  No fault,
 * no hang. */
kvc_status kvc_selftest_bounded_wait(void* workspace, uint64_t limit_ns, void* stream);

/* ---- Device-resident lengths: graph-capturable decode steps -------------
 *
 * "16. Prefill, decode and the KV cache", the cache protocol paragraph after
 * "Design choices worth noticing": a static cache lets a step be captured in
 * a CUDA graph.  A captured step must take nothing from the host that changes
 * per step, so while these calls are in use the lengths live in a caller-owned
 * device array and the step's work partition is computed on the device.
 *
 * Bytes of that array: int32 [layers][B]. */
size_t kvc_device_lens_bytes(const kvc_cache* c);

/* Copy the host lengths into dev_lens (caller-owned device memory of
 * kvc_device_lens_bytes(c) bytes, 4-byte aligned; synchronizes `stream`) and
 * hand them over to the device: from now on kvc_decode_step reads and
 * advances them, and every call that reads or writes the host lengths
 * (append, attention, truncate, reset, set/get lens, length, noalloc)
 * returns KVC_ERR_ARG until kvc_lens_from_device.  dev_lens must stay valid
 * until then. */
kvc_status kvc_lens_to_device(kvc_cache* c, int32_t* dev_lens, void* stream);

/* Copy the device lengths back to the host (synchronizes `stream`) and make
 * the host copy authoritative again.  KVC_ERR_ARG if the lengths are not on
 * the device, or if a device length lies outside 0..max_len (then they stay
 * on the device). */
kvc_status kvc_lens_from_device(kvc_cache* c, void* stream);

/* One step of kvc_append_attention with the lengths on the device: appends
 * n_new[b] rows of k_new / v_new [B, Hkv, T, d] at row b's device length, then
 * the T queries q [B, Hq, T, d] attend exactly as in kvc_gqa_attention, and
 * the device lengths advance by n_new.  n_new is a device int32 [B].  bf16
 * and FP8 caches of d = 128, and bf16 caches of d = 64, with G * T <= 16 query
 * rows per KV head (decode and short verify).
 * Three kernels are enqueued (device plan, attention with the append fused
 * in, combine), with nothing read from the host that changes per step, so
 * the call can be captured in a CUDA graph and replayed with new contents of
 * q, k_new, v_new and n_new.  The workspace is the one kvc_workspace_bytes
 * sizes (plus its device plan region, included there).
 * Errors found on the host (nothing enqueued): KVC_ERR_ARG (lengths on the
 * host, pointers, dtype), KVC_ERR_SHAPE (G * T > 16, Hq % Hkv), KVC_ERR_WORKSPACE,
 * KVC_ERR_CUDA.  A row with n_new[b] outside 0..T or past max_len rejects the
 * whole step on the device: nothing is written, no length changes, and the
 * next kvc_device_status returns KVC_ERR_OVERFLOW. */
kvc_status kvc_decode_step(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new, int q_heads,
                           int T, const int32_t* n_new, void* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Number of kernels this handle has enqueued so far (append, attention and,
 * when a call's units were split across CTAs, the combine kernel).  Host
 * counter only; lets a caller check how many launches a region issued. */
uint64_t kvc_kernel_launches(const kvc_cache* c);

/* Message of the calling thread's last failed call ("" if none). */
const char* kvc_last_error(void);

/* Library version string. */
const char* kvc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
