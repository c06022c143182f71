/*
 * kvarn.h -- C ABI of the KVarN KV-cache library for NVIDIA GB300 (sm_103a).
 *
 * KVarN ("KVarN: Variance-Normalized KV-Cache Quantization Mitigates Error
 * Accumulation in Reasoning Tasks"; fig1.dev summary, "What it is") stores the
 * K/V cache of each attention layer in three regions (anbeeld.com, "KVarN KV
 * Cache: Implementation and Benchmarks", section 2.1):
 *   - the sink: the first 128 tokens, kept exact (fp16) for good;
 *   - sealed groups: every later run of 128 tokens is, when its last token
 *     arrives, rotated by a Hadamard matrix over head_dim, variance-normalised by
 *     16 Sinkhorn iterations over the token and channel axes, rounded to nearest
 *     at b bits, and stored as one packed record per (group, KV head, K|V);
 *   - the tail: the partial newest group, kept exact (fp16) until it fills.
 * Decode attention rotates the query by the same matrix, reads the sink and the
 * tail exact and every sealed record directly, and rotates the output back once
 * per token (anbeeld.com, section 1).
 *
 * Record format (one 128 x 128 group matrix; all multi-byte fields little-endian;
 * size 528 + 2048*b bytes, a multiple of 16):
 *   [0,4)     delta, f32    step of the quantisation grid
 *   [4,8)     m, f32        minimum of the grid
 *   [8,16)    zero
 *   [16,272)  a[128], f16   per-token Sinkhorn scale
 *   [272,528) c[128], f16   per-channel Sinkhorn scale
 *   [528,...) codes, b bits each, packed least-significant first into 32-bit
 *             words; K codes token-major (token i, then channel j), V codes
 *             channel-major (channel j, then token i).
 * Dequantised, rotated frame: yhat_ij = a_i * c_j * (m + delta * q_ij); original
 * frame: xhat = yhat * H with H the Sylvester Hadamard matrix scaled by 1/sqrt(128).
 *
 * Conventions for every call below:
 *   - Memory: the caller allocates the device memory of the cache (one block,
 *     sized by kvarn_cache_required_bytes) and every q/k/v/out buffer. No call
 *     allocates or frees device memory. Host pointers are marked "host". A buffer
 *     marked "device" may also be pinned host memory that kernels reach at the same
 *     address (cudaHostAlloc under unified addressing; on Grace systems the GPU reads
 *     and writes it over NVLink-C2C): the kernels then move the data themselves.
 *     kvarn_device_accessible tells which pointers qualify.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls enqueue work and return without synchronising. All calls on
 *     one cache handle must be ordered on the GPU (issue them to one stream):
 *     they share the split-K workspace.
 *   - Errors: arguments are checked on the host before anything is enqueued; a
 *     call that returns an error other than KVARN_ECUDA leaves the cache state
 *     unchanged. KVARN_ECUDA reports a failed CUDA call or launch; the message is
 *     kept per thread (kvarn_last_error). A failure detected inside a kernel (a
 *     wait that gave up) is recorded in the cache's device error word and is
 *     returned by kvarn_check_device_error after the stream has been synchronised.
 *   - Threads: a handle is not thread-safe; use one handle per host thread.
 *   - Sizes: head_dim, group size and sink length are 128; bits per side are
 *     2, 4 or 8 in any K/V pair; 3, 5 or 6 with K and V alike (kvarn3, kvarn5, kvarn6);
 *     or the pairs K6/V5, K5/V4, K3/V2 (anbeeld.com sections 4-6 name these widths and
 *     presets); the number of query heads per KV head is 1, 2 or 4 (query head h
 *     reads KV head h / (num_q_heads / num_kv_heads)).
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvarn_cache kvarn_cache;

typedef enum {
    KVARN_OK = 0,
    KVARN_EINVAL = 1,    /* bad argument: id, size, bit width, null pointer */
    KVARN_ENOMEM = 2,    /* the device block passed to kvarn_cache_create is too small */
    KVARN_ECAPACITY = 3, /* pool of sealed-group slots, max_seq_len or per-call limit exceeded */
    KVARN_ECUDA = 4,     /* a CUDA call or kernel launch failed */
    KVARN_ESTATE = 5,    /* the call does not fit the sequence's state (e.g. no such group yet) */
    KVARN_ETIMEOUT = 6   /* a bounded wait inside a kernel gave up (see kvarn_check_device_error) */
} kvarn_status;

/* Flags for kvarn_config.flags. */
#define KVARN_FLAG_HOST_ONLY 1 /* bookkeeping only: no CUDA call and no launch is made.
                                  For testing the cache logic on machines without a GPU. */
#define KVARN_FLAG_TEST_STALL 2 /* testing the timeout path only: in every decode launch one
                                   thread waits, before any copy is issued, on a word that
                                   nothing sets; the bounded wait gives up after about 2 s,
                                   records the timeout in the error word and the launch goes
                                   on (its results stay correct). kvarn_check_device_error
                                   then returns KVARN_ETIMEOUT. Not for production use. */

typedef struct {
    int32_t num_layers;     /* attention layers held by this cache */
    int32_t max_seqs;       /* sequence ids are 0 .. max_seqs-1 */
    int32_t num_q_heads;    /* Hq */
    int32_t num_kv_heads;   /* Hkv; Hq / Hkv in {1, 2, 4} */
    int32_t head_dim;       /* must be 128 */
    int32_t k_bits;         /* bits per K code: 2, 3, 4, 5, 6 or 8 (see Sizes above) */
    int32_t v_bits;         /* bits per V code: 2, 3, 4, 5, 6 or 8 (see Sizes above) */
    int32_t group_size;     /* must be 128 (anbeeld.com 2.1) */
    int32_t sink_tokens;    /* must be 128 (anbeeld.com 2.1) */
    int32_t sinkhorn_iters; /* 16 in the method (anbeeld.com 1); 0..64 accepted */
    int32_t max_seq_len;    /* longest sequence, tokens */
    int32_t pool_groups;    /* slots in the sealed-group pool; one slot holds one
                               (sequence, layer, group) for all KV heads, K and V */
    int32_t flags;          /* KVARN_FLAG_* */
    int32_t tail_floor;     /* groups of recent tokens kept exact beyond the partial one:
                               0 = the published design (the tail is the partial newest
                               group, 0..127 tokens); F = 1..3 = a floor of F groups, as
                               BeeLlama does with F = 1 (anbeeld.com 2.1): group g is sealed
                               when group g + F fills, so once the body starts at least
                               128 F recent tokens stay exact (the tail holds 128 F ..
                               128 F + 127 of them) */
} kvarn_config;

typedef struct {
    uint64_t device_bytes;          /* bytes of the device block the cache uses */
    uint64_t record_bytes_k;        /* one sealed K group matrix */
    uint64_t record_bytes_v;        /* one sealed V group matrix */
    uint64_t slot_bytes;            /* one pool slot (all KV heads, K and V) */
    uint64_t pool_slots_total;
    uint64_t pool_slots_used;
    uint64_t tokens_cached;         /* sum of lengths over sequences and layers */
    uint64_t sealed_tokens;         /* tokens held in sealed groups */
    uint64_t exact_tokens;          /* tokens held exact (sink + tail) */
    uint64_t sealed_bytes;          /* record bytes in use */
    uint64_t exact_bytes;           /* fp16 bytes of the exact tokens held */
    double body_bits_per_element;   /* sealed record bits / sealed elements, K and V averaged */
    double all_in_bits_per_element; /* (sealed + exact bytes) * 8 / cached elements */
} kvarn_stats;

/* Size of a record for one 128 x 128 group matrix at `bits` bits (528 + 2048*bits),
 * or 0 for an unsupported width. */
size_t kvarn_record_bytes(int32_t bits);

/* Bytes of device memory kvarn_cache_create needs for `cfg`. EINVAL on a bad config. */
kvarn_status kvarn_cache_required_bytes(const kvarn_config* cfg, size_t* bytes);

/* Create a cache in caller-owned device memory `dev_mem` (at least
 * kvarn_cache_required_bytes, 256-byte aligned). The handle (host memory) is
 * written to *out. Every sequence starts empty. The device block is initialised
 * lazily by the first call that enqueues work. ENOMEM if `bytes` is too small. */
kvarn_status kvarn_cache_create(const kvarn_config* cfg, void* dev_mem, size_t bytes, kvarn_cache** out);

/* Free the host handle. The device block stays the caller's. NULL is ignored. */
void kvarn_cache_destroy(kvarn_cache* cache);

/* Append n_tokens[i] tokens to sequence seq_ids[i] of `layer`, for i < n_seqs
 * (anbeeld.com 2.1). k, v: device fp16, [sum(n_tokens)][num_kv_heads][128], the
 * sequences' tokens back to back in the order of seq_ids, post-RoPE and unrotated.
 * Tokens at positions < 128 go to the sink; each body group that fills is sealed
 * (rotation, 16 Sinkhorn iterations, rounding, packing) into a newly taken pool
 * slot; the rest go to the tail. seq_ids, n_tokens: host arrays. ECAPACITY (state
 * unchanged) if the pool or max_seq_len would overflow. Duplicate seq ids: EINVAL. */
kvarn_status kvarn_append(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                          const int32_t* n_tokens, const void* k, const void* v, void* stream);

/* Decode attention of one query token per sequence over the whole cached
 * sequence (sink exact, sealed groups from their records, tail exact), with the
 * query rotated in and the sealed part of the output rotated back once
 * (anbeeld.com 1 and 2.1). q: device fp16 [n_seqs][num_q_heads][128];
 * out: device fp16 [n_seqs][num_q_heads][128]; softmax_scale is applied to q.k
 * (usually 1/sqrt(128)). Empty sequences give zero output. n_seqs <= 256. */
kvarn_status kvarn_decode_attention(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                    const void* q, void* out, float softmax_scale, void* stream);

/* One decode step in a single kernel launch: append one token per sequence
 * (k, v: device fp16 [n_seqs][num_kv_heads][128]), seal the group that this token
 * completes, if any (before the attention reads it: the group is quantised "at the
 * moment its last token arrives", anbeeld.com 2.1), then decode attention as in
 * kvarn_decode_attention, the query seeing every token including the new one.
 * Results equal kvarn_append(1 token each) followed by kvarn_decode_attention. */
kvarn_status kvarn_decode_step(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                               const void* k, const void* v, const void* q, void* out, float softmax_scale,
                               void* stream);

/* Prefill (many-query) attention: the queries of the last q_lens[i] tokens of
 * sequence seq_ids[i] (positions n - q_lens[i] .. n - 1, n its current length), each
 * attending causally to the cached keys at positions up to its own. The cache is read
 * as it stands (sink and tail exact; sealed groups from their records, the query
 * rotated in and the sealed part rotated back, anbeeld.com 1 and 2.1), so a chunk
 * appended by kvarn_append and then attended with this call reads its own tokens
 * sealed wherever their group was sealed by that append.
 * q: device fp16 [sum(q_lens)][num_q_heads][128], the sequences' query rows back to
 * back in the order of seq_ids; out: device fp16, same shape (written, not read).
 * seq_ids, q_lens: host arrays; 0 <= q_lens[i] <= n; n_seqs <= 256. EINVAL (nothing
 * enqueued) on bad ids, lengths or pointers; sum(q_lens) * num_q_heads < 2^31. */
kvarn_status kvarn_prefill_attention(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                     const int32_t* q_lens, const void* q, void* out, float softmax_scale,
                                     void* stream);

/* Prefill of a prompt chunk: kvarn_append(n_tokens, k, v) (which seals every group the
 * chunk completes, many per launch) followed by kvarn_prefill_attention with
 * q_lens = n_tokens. Arguments of both are checked before anything is enqueued. */
kvarn_status kvarn_prefill(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                           const int32_t* n_tokens, const void* k, const void* v, const void* q, void* out,
                           float softmax_scale, void* stream);

/* Decode attention as kvarn_decode_attention, for callers that cannot allocate device
 * memory: a plugin inside a serving engine that owns all device memory through its own
 * pool and forbids cudaMalloc, or a process under a hard device-memory cap, still has
 * the cache's block and its q/out buffers, but cannot get a fresh allocation for the
 * split-K scratch (partial softmax states). This call places that scratch in a fixed
 * static device array of the library instead; it allocates and frees nothing.
 * The KVarN pages have no counterpart of this call; it is an interface addition.
 * Limit: max_seqs * num_kv_heads of the cache <= 128 (the array holds 128 blocks of
 * 32 partial states, 8.7 MB per GPU, kept until the process exits); a larger cache is
 * rejected with KVARN_ECAPACITY and a message in kvarn_last_error.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture. The
 * current device must be the one that holds the cache (EINVAL otherwise): each device
 * has its own copy of the array.
 * Every call reuses the partial states left by the previous call (each call tags its own
 * with a fresh epoch), so calls that overlap on the GPU (other streams, other caches,
 * other threads) race: order them on one stream. */
kvarn_status kvarn_decode_attention_noalloc(kvarn_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                            const void* q, void* out, float softmax_scale, void* stream);

/* Convert one sealed group matrix to a standard layout ("others convert to a
 * standard cache layout first", anbeeld.com 2.1): out = yhat (frame 1, rotated) or
 * yhat * H (frame 0, original), [128 tokens][128 channels], fp32 if out_fp32 else
 * fp16. which: 0 = K, 1 = V. ESTATE if the group is not sealed. */
kvarn_status kvarn_dequant_group(kvarn_cache* cache, int32_t layer, int32_t seq_id, int32_t group,
                                 int32_t kv_head, int32_t which, int32_t frame, int32_t out_fp32, void* out,
                                 void* stream);

/* Snapshot of a cache (checkpoint and restore). The KVarN pages have no counterpart of
 * these calls; they are an interface addition for serving (moving or parking a cache).
 * A snapshot holds the host bookkeeping (sequence lengths, block table) and the device
 * state that attention reads: the exact sink and tail regions of every sequence and the
 * pool slots in use (records of every sealed group), in one host byte image with a
 * versioned header that records the cache's configuration.
 * kvarn_snapshot_bytes: size of the image of the cache's current state.
 * kvarn_snapshot_save: write the image into host memory `dst` (pageable or pinned, at
 * least kvarn_snapshot_bytes). It is ordered after the work already enqueued on `stream`
 * and returns once the copies are complete (the stream is synchronised); work on other
 * streams that writes the cache must be complete before the call.
 * kvarn_snapshot_load: replace the whole state of `cache` (created with the same
 * configuration; flags may differ) by the image at `src`. The image is checked first
 * (header, configuration, sizes, every table entry in range, no slot used twice, each
 * sequence's sealed groups exactly those its length implies): EINVAL leaves the cache
 * unchanged. Returns after the copies are complete. After a load, every call gives the
 * results the saved cache would have given, bit for bit. With KVARN_FLAG_HOST_ONLY no
 * device memory is touched: device sections are written as zeros and skipped on load. */
kvarn_status kvarn_snapshot_bytes(const kvarn_cache* cache, size_t* bytes);
kvarn_status kvarn_snapshot_save(kvarn_cache* cache, void* dst, size_t bytes, void* stream);
kvarn_status kvarn_snapshot_load(kvarn_cache* cache, const void* src, size_t bytes, void* stream);

/* Drop a sequence in every layer and return its pool slots. */
kvarn_status kvarn_seq_release(kvarn_cache* cache, int32_t seq_id);

/* Number of tokens of `seq_id` cached in `layer` (host mirror; no device access). */
kvarn_status kvarn_seq_length(const kvarn_cache* cache, int32_t layer, int32_t seq_id, int64_t* len);

/* Device address and size of the record of (layer, seq, group, kv_head, which). */
kvarn_status kvarn_group_record(const kvarn_cache* cache, int32_t layer, int32_t seq_id, int32_t group,
                                int32_t kv_head, int32_t which, const void** dev_ptr, size_t* bytes);

/* Device addresses of the exact regions of (layer, seq): fp16 [kv_head][128][128]
 * for the sink K/V and [kv_head][128 (tail_floor + 1)][128] for the tail K/V (a ring:
 * tail slot = (position - 128) mod (128 (tail_floor + 1))). */
kvarn_status kvarn_exact_regions(const kvarn_cache* cache, int32_t layer, int32_t seq_id, const void** sink_k,
                                 const void** sink_v, const void** tail_k, const void** tail_v);

/* Sizes and bits per element (fig1.dev "Why it matters": about 2.3 at two bits). */
kvarn_status kvarn_cache_stats(const kvarn_cache* cache, kvarn_stats* out);

/* Seal n independent fp16 group matrices x[n][128][128] (token rows) into
 * records[n][kvarn_record_bytes(bits)] with the cache's algorithm; which selects
 * the K (0, token-major) or V (1, channel-major) code order. scales, if not NULL:
 * device f32 [n][256], the Sinkhorn token scales a[128] then channel scales c[128]
 * before their rounding to fp16. All pointers device, 16-byte aligned. */
kvarn_status kvarn_seal_groups(const void* x, int32_t n, int32_t bits, int32_t which, int32_t sinkhorn_iters,
                               void* records, float* scales, void* stream);

/* Partition of a decode call's work over CTAs, the one every decode call uses
 * (exposed to test and inspect schedules; host only, no CUDA call). The work is a
 * line of n_blocks blocks, block k holding units[k] >= 1 scheduling units (one
 * sealed group pair is one unit); the first head[k] units of block k
 * (1 <= head[k] <= units[k]; a decode call's exact part and seal of a (sequence,
 * KV head)) must go whole to one CTA. Writes the cut table cuts[0..n] (host array
 * of max_ctas + 1 entries): cuts[0] = 0, cuts[n] = the total, CTA b takes units
 * [cuts[b], cuts[b + 1]), n <= max_ctas, no range empty, no cut strictly inside a
 * head, every block covered by at most max_span ranges; n in *n_ctas. The cuts are
 * the greedy fill (each cut as late as a bound L and the heads allow) for the
 * smallest L >= min_load found by bisection; a range's cost is its units plus
 * item_cost (>= 0) for every block it touches beyond its first two (a decode CTA
 * builds the query tables of its first two blocks up front; a later block's is built
 * while the CTA's warps wait). With item_cost 0 and when max_span does not bind, no
 * valid partition into max_ctas ranges has a smaller largest range. KVARN_EINVAL for
 * bad arguments, KVARN_ECAPACITY if the total reaches 2^31 or nothing fits. */
kvarn_status kvarn_partition_units(int32_t n_blocks, const int32_t* units, const int32_t* head, int32_t max_ctas,
                                   int32_t max_span, int32_t min_load, int32_t item_cost, int32_t* cuts,
                                   int32_t* n_ctas);

/* Read and clear the device error word of the cache (synchronises `stream`).
 * KVARN_OK; KVARN_ETIMEOUT if a bounded wait in a kernel gave up; KVARN_ESTATE for any
 * other recorded fault: a block-table entry out of range, a block split over too many
 * CTAs, or a split-K partial that the merge needed but that carried another call's
 * epoch (overlapping calls on the shared workspace of kvarn_decode_attention_noalloc);
 * such a partial is left out of the output instead of being mixed in. */
kvarn_status kvarn_check_device_error(kvarn_cache* cache, void* stream);

/* *accessible = 1 if kernels can dereference ptr as given: device or managed memory, or
 * pinned host memory mapped at the same address (see Memory above); 0 otherwise (also
 * for ordinary pageable host memory and unknown pointers). KVARN_ECUDA only if the
 * CUDA runtime cannot answer. Host only; launches nothing. */
kvarn_status kvarn_device_accessible(const void* ptr, int32_t* accessible);

/* Static text for a status code. */
const char* kvarn_status_string(kvarn_status status);

/* Last CUDA error message seen by a call on this thread ("" if none). */
const char* kvarn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
