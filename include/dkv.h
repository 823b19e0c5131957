/*
 * dkv.h — C ABI of the zero-copy host-resident KV-cache attention library.
 *
 * The method is DirectKV ("No Buffer, No Bottleneck: Efficient Zero-Copy KV
 * Cache Offloading for Long-Context LLMs").  Its pieces, as the pages
 * describe them:
 *   - KV Cache Manager: K/V tensors live in pinned host memory allocated with
 *     cudaHostAlloc and are read by GPU kernels through zero-copy pointers;
 *     once written they stay there across decode iterations ("Paper Notes:
 *     DirectKV", System Architecture, KV Cache Manager).
 *   - Attention Fusion Engine: one kernel computes the K/V projection of the
 *     new token(s), keeps the fresh K/V on chip and runs attention over the
 *     host-resident cache (same page, System Architecture and Key Ideas (2)).
 *     Prefill iterates over HBM-resident Q for each host K/V tile; decode
 *     iterates over all cached K/V for the single new query (same page,
 *     System Architecture, prefill/decode strategies).
 *   - CPU-memory-aware tiling: a host K/V tile is fetched once and reused by
 *     every query tile and head that needs it (same page, Key Ideas (1)).
 *   - Kernel Adaptor: picks a precompiled kernel by dtype, head dim, tile and
 *     phase (same page, System Architecture, Kernel Adaptor).
 * The attention computed is softmax(Q.K^T / sqrt(d)).V with K = X.Wk,
 * V = X.Wv (same page, Fundamental Underlying Technologies, Kernel Fusion).
 *
 * Conventions for every call:
 *   - Shapes: B batch, T new tokens per sequence, H hidden, Hq query heads,
 *     Hkv KV heads (Hq a multiple of Hkv; query head h uses KV head
 *     h / (Hq/Hkv)), D head dim.
 *   - x is [B, T, H]; Wq is [H, Hq*D]; Wk and Wv are [H, Hkv*D]; out is
 *     [B, T, Hq, D]; all row-major, all in the cache's dtype, all DEVICE
 *     pointers owned by the caller.
 *   - The K cache and the V cache are each [B][Hkv][max_tokens][D] in pinned,
 *     mapped host memory owned by the library (dense caches; paged caches
 *     hold pools of pages, layered caches one such pair per layer, see
 *     their allocators).  Elements are the dtype, or 8-bit E4M3 for caches
 *     allocated with that format.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Work is enqueued; nothing waits for the GPU unless
 *     the call says so.
 *   - No call throws.  Argument, capacity and support errors return before
 *     anything is enqueued and leave the cache unchanged.  dkv_last_error()
 *     gives a thread-local detail string for the last failure.
 */
#ifndef DKV_H
#define DKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DKV_OK = 0,
    DKV_ERR_INVALID_ARG = 1,      /* null pointer, bad size, bad handle */
    DKV_ERR_UNSUPPORTED = 2,      /* no precompiled kernel for (dtype, D, G), or a
                                     call that this kind of cache does not serve */
    DKV_ERR_CAPACITY = 3,         /* length + T would exceed max_tokens, or a row
                                     of a paged cache has no page */
    DKV_ERR_NO_MAPPED_MEMORY = 4, /* the device cannot map host memory */
    DKV_ERR_ALLOC = 5,            /* pinned host or device allocation failed */
    DKV_ERR_CUDA = 6,             /* a CUDA runtime call failed */
    DKV_ERR_TIMEOUT = 7           /* a bounded device-side wait gave up */
} dkv_status;

typedef enum { DKV_BF16 = 0, DKV_FP16 = 1 } dkv_dtype;

typedef struct dkv_cache dkv_cache; /* opaque; tagged so a stale handle is rejected */

/* What the cache stores per K/V element: the dtype itself (2 bytes), or 8-bit
 * E4M3 (OCP 8-bit floating point; 1 sign, 4 exponent, 3 mantissa bits; no
 * infinities; largest finite 448), unscaled and saturating.  E4M3 halves the
 * bytes the attention reads across the host link (the FP8 KV cache that
 * "KV Offloading and Transfer" lists among the cheaper things to do first,
 * in section 6, When it's worth it; not part of DirectKV's pages).  New
 * rows are the fp32 projection sums rounded once to E4M3 (to nearest, ties
 * to even, saturating); decode only, bf16 activations only. */
typedef enum { DKV_KV_NATIVE = 0, DKV_KV_E4M3 = 1 } dkv_kv_format;

/* Everything a cache can be: dense (page_tokens 0), paged (page_tokens > 0,
 * one layer), layered (layers > 1, dense), in either element format.
 * layers 0 counts as 1. */
typedef struct {
    int batch, n_kv_heads, head_dim, max_tokens;
    dkv_dtype dtype;
    dkv_kv_format kv_format;
    int layers;
    int page_tokens, num_pages, max_pages_per_seq;
} dkv_cache_desc_t;

/* Sizes of what a cache holds (the pages' memory accounting: zero bytes of
 * HBM staging; "Paper Notes: DirectKV", Experiments, GPU memory). */
typedef struct {
    size_t host_pinned_bytes;  /* K + V caches in pinned, mapped host memory */
    size_t device_workspace_bytes; /* library-owned HBM for q, fresh K/V, partials */
    size_t device_staging_bytes;   /* HBM copies of the cache: always 0 */
    int batch, n_kv_heads, head_dim, max_tokens, dtype;
    int page_tokens;        /* paged caches: rows per page; 0 for a dense cache */
    int num_pages;          /* paged caches: pages in each of the K and V pools */
    int max_pages_per_seq;  /* paged caches: page-table entries per sequence */
    int layers;             /* layered caches: layers held (1 otherwise) */
    int kv_format;          /* dkv_kv_format of the K/V elements */
    int numa_node_wanted;   /* host NUMA node attached to the cache's GPU (-1: unknown) */
    int numa_node;          /* node holding the cache's first page (-1: unknown) */
} dkv_cache_info_t;

/* Allocate a K cache and a V cache of [batch][n_kv_heads][max_tokens][head_dim]
 * elements each with cudaHostAlloc(Mapped | Portable) and obtain their device
 * aliases with cudaHostGetDevicePointer (KV Cache Manager, "Paper Notes:
 * DirectKV", System Architecture).  Sequence lengths start at 0.  The current
 * CUDA device is the one the cache serves.  Host contents are zeroed.
 * Errors: INVALID_ARG (null out, non-positive size, dtype), UNSUPPORTED
 * (head_dim not 64 or 128), NO_MAPPED_MEMORY (device cannot map host
 * memory), ALLOC. */
dkv_status dkv_cache_alloc(dkv_cache** out, int batch, int n_kv_heads, int head_dim,
                           int max_tokens, dkv_dtype dtype);

/* The general allocator behind dkv_cache_alloc, dkv_cache_alloc_layered and
 * dkv_cache_alloc_paged, which also takes the element format.  An E4M3 cache
 * serves dkv_decode / dkv_decode_layer / dkv_decode_unfused / captured steps
 * (its host views hold uint8 E4M3 bits); dkv_prefill, dkv_decode_staged,
 * dkv_prefill_staged and dkv_attend_naive return UNSUPPORTED for it.  Errors: as the three
 * allocators, plus INVALID_ARG for an unknown format, UNSUPPORTED for E4M3
 * with fp16 activations or a paged cache of several layers. */
dkv_status dkv_cache_alloc_ex(dkv_cache** out, const dkv_cache_desc_t* desc);

/* A layered cache: one pinned allocation each for K and V holding `layers`
 * caches of [batch][n_kv_heads][max_tokens][head_dim] back to back, the
 * (layers, batch, heads, tokens, head_dim) host tensor of a whole model
 * ("DirectKV Guide: Zero-Copy KV Offloading on GH200 & GB200", Production
 * Engineering Playbook (1)).  Layers share the sequence lengths: a token's
 * calls go layer 0 .. layers-1 (dkv_decode_layer / dkv_prefill_layer), each
 * appending at the current length, and the lengths advance with the call for
 * the last layer.  dkv_decode / dkv_prefill refuse a layered cache
 * (INVALID_ARG); the measurement baselines need a one-layer cache.
 * Errors: as dkv_cache_alloc, plus INVALID_ARG for layers outside [1, 1024]. */
dkv_status dkv_cache_alloc_layered(dkv_cache** out, int layers, int batch, int n_kv_heads,
                                   int head_dim, int max_tokens, dkv_dtype dtype);

/* A paged cache: K and V pools of [num_pages][n_kv_heads][page_tokens][head_dim]
 * elements each in pinned, mapped host memory, addressed through a per-
 * sequence page table (the KV cache pages that the GPU kernels dereference in
 * place, "DirectKV Guide: Zero-Copy KV Offloading on GH200 & GB200", The
 * DirectKV Architecture (Zero-Copy Page Management) and End-to-End
 * Implementation (the page manager, 16-token pages)).  Logical row t of
 * sequence b lives in pool page table[b][t / page_tokens], row t % page_tokens.
 * Every decode / prefill call works on paged caches exactly as on dense ones;
 * a sequence holds at most max_pages_per_seq * page_tokens rows (its
 * max_tokens).  The page table starts empty (every entry -1).
 * Errors: as dkv_cache_alloc, plus INVALID_ARG when page_tokens is not a power
 * of two in [1, 4096] or num_pages / max_pages_per_seq is not positive. */
dkv_status dkv_cache_alloc_paged(dkv_cache** out, int batch, int n_kv_heads, int head_dim,
                                 int page_tokens, int num_pages, int max_pages_per_seq,
                                 dkv_dtype dtype);

/* Replace a paged cache's page table: table is host memory of
 * [batch][max_pages_per_seq] int32 pool page indices, -1 for none.  The
 * library keeps a host copy (each call checks that the rows it reads and
 * appends, [0, len + T) of every sequence, sit on pages: CAPACITY otherwise)
 * and a device copy, written after the cache's last stream has finished.
 * Pages may be shared between sequences for reading; the caller must not
 * let two sequences append into the same page row.
 * Errors: INVALID_ARG (dense cache, entry outside [-1, num_pages)), CUDA. */
dkv_status dkv_cache_set_page_table(dkv_cache* cache, const int32_t* table);

/* Release the pinned caches and the device workspace.  The caller must make
 * sure no enqueued work still uses the cache.  A handle already freed (or
 * never returned by dkv_cache_alloc) gives INVALID_ARG. */
dkv_status dkv_free(dkv_cache* cache);

/* The host NUMA node sysfs reports for a PCI device, given its bus id as
 * cudaDeviceGetPCIBusId prints it ("0000:1B:00.0"), read from
 * <sysfs_root>/bus/pci/devices/<id>/numa_node (sysfs_root null or "": /sys);
 * -1 when unknown, absent or malformed.  Every cache allocation pins its pages
 * with the calling thread's memory policy preferring the node of the current
 * GPU (so each replica's cache sits next to its own host link; "Paper Notes:
 * DirectKV", System Architecture, KV Cache Manager), then restores the policy;
 * DKV_NUMA=0 in the environment turns that off.  dkv_cache_info reports the
 * node wanted and the node the first page landed on. */
int dkv_pci_numa_node(const char* pci_bus_id, const char* sysfs_root);

/* Allocates and touches one page of ordinary host memory with the calling
 * thread's policy preferring `node`, as the cache allocation does, and
 * returns the node it landed on (-1 if unknown).  Needs no GPU. */
int dkv_numa_probe(int node);

/* Host addresses of the two caches ([B][Hkv][max_tokens][D] each), for
 * filling prefixes and reading back appended rows.  The host must not touch
 * rows that enqueued work reads or writes until that work has finished. */
dkv_status dkv_cache_host_ptrs(dkv_cache* cache, void** k_host, void** v_host);

/* Device aliases of the same two caches (zero-copy pointers). */
dkv_status dkv_cache_device_ptrs(dkv_cache* cache, void** k_dev, void** v_dev);

/* Set / read the per-sequence lengths (cached rows per sequence), len[B].
 * Set: INVALID_ARG if a length is negative, CAPACITY if above max_tokens. */
dkv_status dkv_cache_set_lengths(dkv_cache* cache, const int32_t* len);
dkv_status dkv_cache_get_lengths(const dkv_cache* cache, int32_t* len);

dkv_status dkv_cache_info(const dkv_cache* cache, dkv_cache_info_t* info);

/* Reserve the device workspace for calls with up to n_q_heads query heads and
 * up to max_new_tokens new tokens per sequence, so that later calls allocate
 * nothing.  Without it the first call of a larger shape grows the workspace
 * (a cudaMalloc on the calling thread, after synchronising the cache's last
 * stream). */
dkv_status dkv_cache_reserve(dkv_cache* cache, int n_q_heads, int max_new_tokens);

/* One decode step (T = 1) for every sequence: q = x.Wq, k = x.Wk, v = x.Wv
 * (fp32 accumulation in sequential order over H, rounded to the dtype), the
 * new k, v appended at row len[b] of the host cache, then softmax attention
 * of the Hq query heads over keys 0..len[b] of their KV head (the new token
 * included), written to out [B, 1, Hq, D].  Lengths advance by 1 when the
 * call is enqueued.  One cooperative launch of the fused kernel plus a
 * split-KV combine launch.  With an E4M3 cache the new k, v are the fp32
 * sums rounded once to E4M3 and the attention reads the decoded E4M3 rows.
 * Errors: INVALID_ARG (also for a layered cache: use dkv_decode_layer),
 * UNSUPPORTED (dtype, D, Hq/Hkv), CAPACITY, ALLOC (workspace growth), CUDA.
 * Device-side wait timeouts are reported by dkv_sync_status. */
dkv_status dkv_decode(dkv_cache* cache, const void* x, const void* wq, const void* wk,
                      const void* wv, int hidden, int n_q_heads, void* out, void* stream);

/* dkv_decode for one layer of a layered cache (layer 0 of any other cache):
 * x, W and out are that layer's; the append goes to the layer's cache at the
 * current length, and the lengths advance after the last layer.  Errors: as
 * dkv_decode, plus INVALID_ARG for a layer outside [0, layers). */
dkv_status dkv_decode_layer(dkv_cache* cache, int layer, const void* x, const void* wq,
                            const void* wk, const void* wv, int hidden, int n_q_heads, void* out,
                            void* stream);

/* Capture one whole decode step (every layer in order, then the lengths
 * advance by one) into a CUDA graph held by the cache, so that a step costs
 * one graph launch instead of two launches per layer.  x, wq, wk, wv, out are
 * host arrays of `layers` device pointers (as dkv_decode_layer takes them);
 * the graph keeps those pointers and the kernel configuration chosen now, and
 * reads the sequence lengths from device memory at run time, so every launch
 * appends at the lengths of its own step.  Captures on a stream of the
 * library's own; replaces an earlier capture.  A later call that needs a
 * larger workspace (a longer prefill, say) discards the capture, since the
 * graph holds workspace addresses; dkv_step_graph_launch then returns
 * INVALID_ARG until the step is captured again.  Errors: as dkv_decode, CUDA
 * (the capture or instantiation failed). */
dkv_status dkv_step_graph_capture(dkv_cache* cache, int hidden, int n_q_heads,
                                  const void* const* x, const void* const* wq,
                                  const void* const* wk, const void* const* wv,
                                  void* const* out);

/* Launch the captured step on `stream`: checks capacity (CAPACITY if a
 * sequence is full), publishes the host lengths to the device first if they
 * changed outside graph steps (one synchronisation), then launches and
 * advances the host lengths.  INVALID_ARG if nothing was captured. */
dkv_status dkv_step_graph_launch(dkv_cache* cache, void* stream);

/* One prefill (chunked-prefill) call: T new tokens per sequence at rows
 * [len[b], len[b]+T).  Query t of sequence b (absolute position len[b]+t)
 * attends causally to keys 0..len[b]+t.  Q = x.Wq is written to HBM first
 * (Q is HBM-resident, "Paper Notes: DirectKV", System Architecture, prefill
 * strategy); the fused kernel then holds each host K/V chunk stationary in
 * shared memory, computing the fresh K/V rows of chunks in the new region
 * in place and appending them to the host cache, and runs every query tile
 * of the KV head against it; a combine launch merges the per-chunk partial
 * results.  out is [B, T, Hq, D].  Lengths advance by T when enqueued.
 * Errors as dkv_decode, plus UNSUPPORTED for an E4M3 cache. */
dkv_status dkv_prefill(dkv_cache* cache, const void* x, int T, const void* wq, const void* wk,
                       const void* wv, int hidden, int n_q_heads, void* out, void* stream);

/* dkv_prefill for one layer of a layered cache (layer 0 of any other cache);
 * the lengths advance by T after the last layer. */
dkv_status dkv_prefill_layer(dkv_cache* cache, int layer, const void* x, int T, const void* wq,
                             const void* wk, const void* wv, int hidden, int n_q_heads, void* out,
                             void* stream);

/* Synchronise the stream, then return and clear the device status word that
 * bounded waits write (DKV_ERR_TIMEOUT), or DKV_ERR_CUDA if the stream
 * reported an error.  The word stays set until this call reads it: the
 * combine kernels of every decode or prefill enqueued while it is set write
 * NaN outputs instead of merging partials that were never written. */
dkv_status dkv_sync_status(dkv_cache* cache, void* stream);

/* Tuning overrides for ablations; 0 keeps the adaptor's choice.
 *   splits       decode: key-range splits per (sequence, KV head)
 *   tile_n       keys per host tile (decode) or per stationary chunk (prefill)
 *   stages       decode ring depth m */
dkv_status dkv_cache_set_tuning(dkv_cache* cache, int splits, int tile_n, int stages);

/* Test hook for the failure-detection path: while enabled, the producer
 * warps of every dkv_decode on this cache never signal their first host tile
 * (and the loader of every dkv_prefill never signals its chunk's host rows),
 * so a bounded wait expires after about one second; the kernel drains its own
 * copies and returns, and dkv_sync_status reports DKV_ERR_TIMEOUT.  The output
 * of such a call is NaN; the cache rows before the append are untouched and
 * the context stays usable. */
dkv_status dkv_cache_debug_withhold(dkv_cache* cache, int enable);

const char* dkv_status_str(dkv_status s);
const char* dkv_last_error(void);

/* Projection Y[M,N] = X[M,K] . W[K,N] on the tensor cores (the Q projection
 * step of dkv_prefill, q = x.Wq; "Paper Notes: DirectKV", Fundamental
 * Underlying Technologies, Kernel Fusion).  Row-major device tensors in
 * `dtype`, fp32 accumulation, one rounding to the dtype.  K must be a
 * multiple of 8 and N of 64; rows past M and columns past N are not
 * touched.  The caller owns all three buffers. */
dkv_status dkv_project(const void* x, const void* w, void* y, int M, int K, int N,
                       dkv_dtype dtype, void* stream);

/* ---- measurement kernels (internal baselines and link probes) ----------- */

/* Stream `bytes` (a multiple of 16) from `src` (a device pointer: a mapped
 * host alias for the link, HBM for the HBM rate) with 16-byte loads across
 * the whole GPU; the folded sum goes to sink[0] (device, 16 bytes) so the
 * loads cannot be elided.  The plain zero-copy streaming kernel whose rate is
 * the host-link denominator of the roofline. */
dkv_status dkv_probe_read(const void* src, size_t bytes, void* sink, void* stream);

/* Write `bytes` (a multiple of 16) of a pattern to `dst` with 16-byte stores. */
dkv_status dkv_probe_write(void* dst, size_t bytes, void* stream);

/* Launch floor: an empty kernel (it reads and writes nothing) launched
 * cooperatively with `grid` CTAs of `threads` threads (a multiple of 32, at
 * most 1024) and `smem_bytes` of dynamic shared memory (at most 227 KB).
 * Timed with CUDA events around it, it gives what launch and completion add
 * to a kernel's measured time.  INVALID_ARG for another shape; a grid that
 * cannot be co-resident is reported as a CUDA error. */
dkv_status dkv_probe_launch(int grid, int threads, int smem_bytes, void* stream);

/* Naive untiled zero-copy decode attention (the pages' "naive zero-copy"
 * baseline, "Paper Notes: DirectKV", Experiments, CPU-aware tiling): one CTA
 * per (sequence, query head, split) reads its KV head's rows straight from
 * the host cache with no shared-memory tile and no reuse across the heads of
 * a group.  It attends q (HBM, [B, Hq, D], the dtype) over keys 0..len[b]-1
 * of the cache as it stands (no projection, no append) into out [B, Hq, D].
 * Dense caches only (UNSUPPORTED for a paged cache). */
dkv_status dkv_attend_naive(dkv_cache* cache, const void* q, int n_q_heads, void* out,
                            void* stream);

/* Separate-kernel baseline (the unfused design the pages compare against,
 * "Paper Notes: DirectKV", Experiments & Results, Fused kernel (Fig. 13), and
 * Key Ideas (2)): the same
 * decode as dkv_decode split into two launches, a projection that writes q to
 * HBM and appends the fresh K/V rows to the host cache, then an attention
 * launch that reads every row, the appended one included, back across the
 * link.  Same arguments, results and errors as dkv_decode. */
dkv_status dkv_decode_unfused(dkv_cache* cache, const void* x, const void* wq, const void* wk,
                              const void* wv, int hidden, int n_q_heads, void* out,
                              void* stream);

/* Copy-to-HBM-then-attend baseline (swap-style staging, "Paper Notes:
 * DirectKV", Motivation): cudaMemcpyAsync the cached rows [0, len[b]) of
 * every (sequence, KV head) into the caller's HBM buffers k_stage, v_stage
 * (each [B][Hkv][max_tokens][D]) and run the same fused decode as dkv_decode
 * reading the prefix from HBM (the append still goes to the host cache).
 * Dense caches only (UNSUPPORTED for a paged cache). */
dkv_status dkv_decode_staged(dkv_cache* cache, const void* x, const void* wq, const void* wk,
                             const void* wv, int hidden, int n_q_heads, void* out,
                             void* k_stage, void* v_stage, void* stream);

/* The same baseline for prefill: cudaMemcpyAsync the cached rows [0, len[b])
 * of every (sequence, KV head) into the caller's HBM buffers k_stage,
 * v_stage (each [B][Hkv][max_tokens][D], device memory the caller owns), then
 * run the same fused prefill as dkv_prefill reading the cached prefix from
 * HBM; the T new rows are still appended to the host cache and the lengths
 * advance by T.  Same arguments, results and errors as dkv_prefill, plus
 * INVALID_ARG for a null staging buffer and UNSUPPORTED for a paged, layered
 * or E4M3 cache. */
dkv_status dkv_prefill_staged(dkv_cache* cache, const void* x, int T, const void* wq,
                              const void* wk, const void* wv, int hidden, int n_q_heads,
                              void* out, void* k_stage, void* v_stage, void* stream);

/* Naive untiled zero-copy prefill (measurement baseline for the pages'
 * CPU-memory-aware tiling, "Paper Notes: DirectKV", Key Ideas (1) and
 * Experiments & Results, Fig. 12).  Same computation, results and append
 * as dkv_prefill, from the same fused kernel, but every (Q tile, chunk)
 * pair gets its own CTA, in the order a Q-stationary kernel streams the
 * chunks, so each chunk of cached rows crosses the host link once per Q tile
 * that sees it instead of once.  The outputs are bit-identical to
 * dkv_prefill's.  Errors as dkv_prefill, plus UNSUPPORTED for a layered or
 * E4M3 cache. */
dkv_status dkv_prefill_naive(dkv_cache* cache, const void* x, int T, const void* wq,
                             const void* wk, const void* wv, int hidden, int n_q_heads,
                             void* out, void* stream);

/* Kernel timing for measurement: when enabled, each dkv_decode / dkv_prefill
 * records a pair of CUDA events on its stream around its main fused kernel
 * (not the projection or combine launches).  dkv_cache_last_kernel_ms waits
 * for the last recorded pair and returns its elapsed time in milliseconds;
 * INVALID_ARG if timing is off or nothing was recorded yet. */
dkv_status dkv_cache_kernel_timing(dkv_cache* cache, int enable);
dkv_status dkv_cache_last_kernel_ms(dkv_cache* cache, float* ms);

/* ---- decode without any allocation -------------------------------------- */

/* The paper has no counterpart to this call; it exists for callers that may
 * not allocate GPU memory at all (code running inside an allocator or
 * memory-pool callback, plug-ins whose host runtime owns every device
 * allocation, services that must hold a fixed memory budget after start-up).
 *
 * Same computation as dkv_decode on caller-owned buffers: q/k/v projection of
 * x, append of the new k, v at row lengths[b] of k_cache / v_cache, attention
 * over rows 0..lengths[b], result in out [B, 1, Hq, D].  k_cache and v_cache
 * are device-accessible pointers to [batch][n_kv_heads][max_tokens][head_dim]
 * caches (normally the mapped aliases of pinned host memory, e.g. from
 * dkv_cache_device_ptrs); lengths is a host array [batch] that this call
 * reads but does not advance.  All tensors are in `dtype`.
 *
 * It calls no cudaMalloc, cudaFree or allocating library routine.  Its
 * scratch (8 MiB: q and fresh K/V workspace, split-KV partials, status word)
 * is a fixed __device__ array that every GPU loading the library holds until
 * the process exits; a shape whose scratch would exceed 8 MiB even with one
 * key-range split is rejected with DKV_ERR_CAPACITY.  Every call on a device
 * shares that array, so calls whose work overlaps on the GPU (other streams,
 * other threads) race and must be serialised by the caller.  The first call
 * on each device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.
 * The address is looked up again on every call (the lookup allocates
 * nothing), so a context that was reset and recreated is served correctly.
 * A device-side wait that gives up (DKV_ERR_TIMEOUT) is recorded in the
 * scratch status word, which every call clears first, and makes the call's
 * outputs NaN; dkv_decode_noalloc_status reads it.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY, CUDA, before anything is
 * enqueued. */
dkv_status dkv_decode_noalloc(const void* x, const void* wq, const void* wk, const void* wv,
                              void* k_cache, void* v_cache, const int32_t* lengths, int batch,
                              int hidden, int n_q_heads, int n_kv_heads, int head_dim,
                              int max_tokens, dkv_dtype dtype, void* out, void* stream);

/* Status of the last dkv_decode_noalloc on the current device, without any
 * allocation: synchronises `stream`, copies the scratch status word into a
 * host variable, clears it if set, and returns DKV_OK or the recorded error
 * (DKV_ERR_TIMEOUT); DKV_ERR_CUDA if the stream reported an error.  Call it
 * after the dkv_decode_noalloc it should report on and before the next one
 * (which clears the word). */
dkv_status dkv_decode_noalloc_status(void* stream);

/* Test hook for the no-allocation path (process-wide): while enabled, the
 * producers of every dkv_decode_noalloc withhold their first tile's signal so
 * that the consumers' bounded wait expires after about a second; the call's
 * outputs are NaN and dkv_decode_noalloc_status reports DKV_ERR_TIMEOUT. */
dkv_status dkv_decode_noalloc_debug_withhold(int enable);

/* Number of kernel launches the last dkv_decode / dkv_prefill enqueued. */
int dkv_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DKV_H */
