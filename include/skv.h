/*
 * skv.h -- C ABI of the sparse-attention KV assembly library (GB300, sm_103a).
 *
 * What the library does.  Long-context decoding keeps the complete KV history
 * of every request in a host memory pool and only a cache of hot tokens on the
 * accelerator; each decode step, per layer, the sparse-attention Top-k indices
 * say which tokens the attention kernel needs, and those tokens are assembled
 * on the device on demand, at token (not page) granularity.  The sources, and
 * the short tags the "Source:" line of each declaration below uses for them:
 *   [talk]   "Sparse Attention-Driven KVCache Management for Domestic AI
 *            Supernodes" (ml-summit.org talk abstract): abstract, and agenda
 *            item 2 (host storage, device cache and index mapping of the
 *            SparseKVCacheManager; the UniDex index-copy operator that keeps
 *            the step graph-executable);
 *   [digest] "SGLang и Tair представили иерархичную Sparse Attention для
 *            хранения полного KV Cache на CPU и экономии GPU-памяти":
 *            paragraph 1 (full KV on the CPU, a Top-k LRU buffer on the GPU),
 *            paragraph 3 (incremental transfer of sparse changes by the Sparse
 *            Diff Kernel, fast I/O kernels);
 *   [xm]     "XM-Sparse: Netpreme X-Mem 突破稀疏注意力吞吐极限": section
 *            "与SGLang HiSparse的集成" (CUDA Graph support; lifecycle publish,
 *            acquire, write back, release), section
 *            "为何稀疏注意力需要快速高容量内存层" (a hot KV buffer in HBM
 *            reduces external-memory reads).
 * Where the pages are silent, a declaration's Source line says so and states
 * the reading this library implements.
 *
 * Geometry.  R request slots, L layers, T_max tokens of pool room per request,
 * rows of row_bytes bytes (576 bf16 = 1152 B for an MLA latent of 512 plus 64
 * rope dims), k Top-k entries per (request, layer) and step, S >= k hot slots
 * per (request, layer).
 *
 * Memory the library owns (all allocated by skv_create, freed by skv_destroy):
 *   pool  [R][L][T_max][row_bytes]  host memory, pinned and mapped into the
 *                                   GPU's address space (the host storage)
 *   hot   [R][L][S][row_bytes]      device memory (the device cache)
 *   tok2slot [R][L][T_max] int32    device; -1 = token not resident
 *   slot2tok [R][L][S] int32        device; -1 = empty slot
 *   ts       [R][L][S] uint32       device; clock of the step that last used the slot (0 = never)
 *   lru      [R][L][S] uint16       device; the S slots ordered by (ts, slot), least recent first
 *   len/active per request, the step clock and the sticky error word -- all
 *   device memory.
 * No call after skv_create allocates; skv_assemble and skv_write_back are
 * therefore safe to capture in a CUDA graph.
 *
 * The replacement rule (the pages name an LRU buffer but not its tie-breaks;
 * these are the readings this library implements):
 *   - a global step clock advances by one on every successful skv_assemble;
 *   - a slot whose token is in this step's Top-k is a hit and is never
 *     evicted in that step;
 *   - the missing tokens, in ascending token order, take the non-hit slots
 *     with the smallest (ts, slot index), in that order;
 *   - every slot used by the step (hits and fills) gets ts = clock.
 *
 * Streams and ordering.  Every call that takes a cudaStream_t only enqueues
 * work on that stream (plus, where stated, a synchronisation of it).  Calls on
 * one context must be ordered: issue them on one stream, or order the streams
 * with events.  Two overlapping calls on one context race.
 *
 * Errors.  Each call returns an skv_status.  Errors that the host can see
 * (bad handle, bad sizes, null pointers, unknown request in skv_release, no
 * free request slot) are returned at once and nothing is enqueued.  Errors
 * that depend on device data (bad request ids in a device array, Top-k entries
 * out of range or repeated, a full pool region) are detected on the device:
 * the call then changes no state, fills its outputs with -1, and ORs an
 * SKV_DEVERR_* bit into a sticky device error word.  While that word is
 * non-zero every later skv_assemble / skv_write_back is a no-op with -1
 * outputs.  skv_get_device_error reads and clears it.  No kernel traps,
 * asserts or spins.
 *
 * Why bad indices and timeouts are device error bits, not skv_status values:
 * they depend on data the host does not see when it enqueues a call (a Top-k
 * tensor produced on the device, a product that has not run yet), and a call
 * must stay stream-ordered and capturable in a CUDA graph, so it cannot wait
 * for them.  They are found on the device and reported through the sticky
 * word; skv_status covers what the host can check when the call is made.
 *
 * Why the configuration gives row_bytes rather than an element count and an
 * element size: the assembly path moves rows as bytes and never reads an
 * element; only skv_attend interprets them, and it requires 576 bf16 (1152
 * bytes).  row_bytes = elements x element size.
 */
#ifndef SKV_H_
#define SKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t / cudaEvent_t without including the CUDA headers (same
 * underlying types). */
typedef struct CUstream_st *skv_stream_t;
typedef struct CUevent_st *skv_event_t;

typedef struct skv_ctx skv_ctx;

/* Every entry point is exported with default visibility; the library is built
 * with everything else hidden. */
#if defined(__GNUC__)
#define SKV_API __attribute__((visibility("default")))
#else
#define SKV_API
#endif

typedef enum {
    SKV_OK = 0,
    SKV_ERR_INVALID_ARG = 1,     /* null pointer, bad size or bad configuration */
    SKV_ERR_OOM = 2,             /* host or device allocation failed in skv_create */
    SKV_ERR_BAD_REQUEST = 3,     /* skv_release / skv_export_*: request id unknown or not active */
    SKV_ERR_NO_FREE_REQUEST = 4, /* skv_publish: all R request slots are in use */
    SKV_ERR_CONTEXT_FULL = 5,    /* skv_publish: T > max_context */
    SKV_ERR_CUDA = 6             /* a CUDA runtime call failed (see skv_last_cuda_error) */
} skv_status;

/* Bits of the sticky device error word. */
#define SKV_DEVERR_BAD_REQUEST 1   /* a request id in [0,R) that is not active, out of range, or repeated in one call */
#define SKV_DEVERR_BAD_INDEX 2     /* a Top-k entry that is neither -1 nor in [0, len of its request) */
#define SKV_DEVERR_DUPLICATE 4     /* a token that appears twice in one (request, layer) Top-k row */
#define SKV_DEVERR_CONTEXT_FULL 8  /* skv_write_back / skv_extend beyond max_context tokens */
#define SKV_DEVERR_TIMEOUT 16      /* skv_attend: a tensor-core product did not complete within its bounded wait */

typedef struct {
    int32_t max_requests;  /* R >= 1: request slots */
    int32_t num_layers;    /* L >= 1 */
    int64_t max_context;   /* T_max >= 1: pool rows per (request, layer) */
    int32_t row_bytes;     /* bytes per KV row; multiple of 16, <= 65536 (1152 for 576 bf16) */
    int32_t topk;          /* k, 1 <= k <= 4096 */
    int32_t hot_slots;     /* S, k <= S <= 16384 */
    int32_t max_batch;     /* largest B of skv_assemble / n of skv_write_back */
    int32_t device;        /* CUDA device ordinal */
} skv_config;

/* Create a context: allocates the pinned, mapped host pool
 * (cudaHostAllocMapped | cudaHostAllocPortable), the device cache and all
 * device state; every request slot starts free and the hot buffer zeroed.
 * Requires R*L*T_max < 2^32 and R*L*S < 2^32.  *out receives the handle.
 * Synchronous.  Returns SKV_ERR_INVALID_ARG for a bad configuration,
 * SKV_ERR_OOM / SKV_ERR_CUDA on allocation failure (nothing is leaked).
 * Source: [talk] agenda item 2 (the SparseKVCacheManager's host storage,
 * device cache and index mapping); [digest] paragraph 1 (full KV on the CPU,
 * a Top-k LRU buffer on the GPU). */
SKV_API skv_status skv_create(const skv_config *cfg, skv_ctx **out);

/* Synchronise the device and free everything.  A null ctx is a no-op.
 * Source: the pages are silent on tearing the manager down; this library's
 * reading is that destroy frees what create allocated, after all enqueued
 * work has finished. */
SKV_API skv_status skv_destroy(skv_ctx *ctx);

/* Publish a request (lifecycle step "publish"): take the lowest free request
 * slot, make its pool region hold T tokens, reset its maps and clocks and zero
 * its hot rows.  rows, if not null, is [L][T][row_bytes] in host or device
 * memory and is copied into the pool; a host source first synchronises
 * `stream` (so in-flight reads of a previously released request finish) and
 * is copied by the CPU.  With rows == null the caller writes the rows in place
 * through skv_pool_rows before the next skv_assemble on this request.  The
 * device reset is enqueued on `stream`.  *out_req receives the id.
 * Errors: SKV_ERR_CONTEXT_FULL (T > max_context), SKV_ERR_NO_FREE_REQUEST.
 * Source: [xm] section "与SGLang HiSparse的集成" (publish). */
SKV_API skv_status skv_publish(skv_ctx *ctx, const void *rows, int64_t T, int32_t *out_req, skv_stream_t stream);

/* Write back one new token per listed request (lifecycle step "write back"):
 * for i < n, for each layer l, rows_dev[i][l][:] is stored into the pool at
 * position len(req_ids_dev[i]) and that length grows by one.  req_ids_dev
 * [n] int32 and rows_dev [n][L][row_bytes] are device memory (rows may also
 * be mapped host memory).  Device-side errors: SKV_DEVERR_BAD_REQUEST
 * (unknown, inactive or repeated id), SKV_DEVERR_CONTEXT_FULL; on error
 * nothing is written.  The new token can be selected from the next
 * skv_assemble on; it is not put into the hot buffer by this call.
 * n == 0 enqueues nothing.  Host errors: n < 0 or n > max_batch, null
 * pointers with n > 0.
 * Source: [xm] section "与SGLang HiSparse的集成" (write back); that the new
 * token enters the pool only, not the hot buffer, is this library's reading
 * (the pages name the step, not its effect on the device cache). */
SKV_API skv_status skv_write_back(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t n, const void *rows_dev,
                          skv_stream_t stream);

/* Extend a request by n tokens at once (the next turn of an agent session:
 * "XM-Sparse: Netpreme X-Mem ...", section "为何稀疏注意力需要快速高容量内存层" --
 * coding agents keep hundreds of sessions and reuse up to 95 % of a session's
 * KV from turn to turn).  rows [L][n][row_bytes] (device memory, or host memory
 * the device can read, 16-byte aligned) are stored into the pool at positions
 * [len, len + n) of every layer and len grows by n.  Unlike release + publish,
 * the request keeps its maps and its hot buffer, so the previous turns' tokens
 * that are still resident keep hitting.  Host errors: SKV_ERR_BAD_REQUEST (not
 * an active request), SKV_ERR_CONTEXT_FULL (n > max_context),
 * SKV_ERR_INVALID_ARG; device error bits: SKV_DEVERR_CONTEXT_FULL when
 * len + n > max_context (nothing written).  n == 0 enqueues nothing. */
SKV_API skv_status skv_extend(skv_ctx *ctx, int32_t req, const void *rows, int64_t n, skv_stream_t stream);

/* One decode step (lifecycle step "acquire"): for each batch entry b < B and
 * layer l, make every token of topk_dev[b][l][0..k) resident in the hot
 * buffer of request req_ids_dev[b], layer l, and write its slot index to
 * slots_dev[b][l][i] (-1 for a -1 entry).  Steps, all on the device:
 *   1. validate ids and entries (nothing changes if any is bad);
 *   2. sparse diff: probe tok2slot; hits keep their slot, misses are
 *      compacted and ordered by token;
 *   3. LRU allocation: the misses take the least recently used non-hit slots
 *      (rule above); evicted tokens leave tok2slot;
 *   4. gather: copy each missed token's row from the host pool into its slot
 *      (16-byte loads through the mapped pool over the host link; steps 2-4
 *      and 5 run in one kernel, one CTA per (b, l), so planning overlaps the
 *      host-link traffic of other units);
 *   5. emit the fixed-shape slot tensor and the per-(b,l) hit and miss counts
 *      (hits_dev / misses_dev [B][L] int32).
 * The hot row of (request r, layer l, slot s) is at
 * skv_hot_buffer() + ((r*L + l)*S + s) * row_bytes.
 * Inputs and outputs are device memory, B <= max_batch.  B == 0 enqueues
 * nothing and does not advance the clock.  Captures into a CUDA graph.
 * Source: [xm] section "与SGLang HiSparse的集成" (acquire; CUDA Graph
 * support); [talk] abstract and agenda items 1-2 (token-level, Top-k-driven
 * assembly; UniDex index copy); [digest] paragraphs 1 and 3 (Top-k LRU
 * buffer; Sparse Diff Kernel).  The tie-break and the order in which misses
 * take victims are this library's reading (the pages give neither). */
SKV_API skv_status skv_assemble(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, const int32_t *topk_dev,
                        int32_t *slots_dev, int32_t *hits_dev, int32_t *misses_dev, skv_stream_t stream);

/* skv_assemble for one layer only: for each batch entry b < B, make every
 * token of topk_dev[b][0..k) resident in the hot buffer of request
 * req_ids_dev[b], layer `layer`, and write its slot to slots_dev[b][i]
 * (hits_dev / misses_dev are [B]).  Other layers are untouched.  A decode
 * step can thus assemble layer by layer, as each layer's Top-k becomes known,
 * and overlap layer l+1's transfer with other work on another stream (the
 * pages: on-demand assembly of the data the current computation needs, its
 * data-movement overhead and HiSparse's prefetching -- "Sparse
 * Attention-Driven KVCache Management for Domestic AI Supernodes", abstract
 * and agenda item 3; "XM-Sparse: Netpreme X-Mem ...", section
 * "与SGLang HiSparse的集成").  Same validation, errors and output conventions as
 * skv_assemble; every successful call advances the step clock by one, so the
 * replacement order within a (request, layer) is the order of the calls that
 * touched it.  Calls on one context must still be ordered (one stream), since
 * they share the control words; the overlap is with the caller's other work.
 * SKV_ERR_INVALID_ARG if layer is outside [0, L).  Captures into a CUDA graph. */
SKV_API skv_status skv_assemble_layer(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, int32_t layer,
                                      const int32_t *topk_dev, int32_t *slots_dev, int32_t *hits_dev,
                                      int32_t *misses_dev, skv_stream_t stream);

/* Prefetch: bring tokens that a coming step is expected to select into the
 * hot buffers ahead of that step, so that its assemble finds them resident
 * and moves fewer rows over the host link while the attention waits (the
 * pages: XM-Sparse keeps HiSparse's prefetching -- "XM-Sparse: Netpreme X-Mem
 * ...", section "与SGLang HiSparse的集成"; the overhead of on-demand data
 * movement -- "Sparse Attention-Driven KVCache Management for Domestic AI
 * Supernodes", agenda item 3).  A prefetch IS an assemble of the candidate
 * tokens whose slot tensor is not returned: the same validation (ids, range,
 * no repeats), the same LRU rule, the same gather, the same clock tick, so a
 * prefetched token counts as used at the prefetch and is the last to be
 * evicted, and the next assemble that selects it is a hit.
 *   layer: -1 for every layer (cand_dev [B][L][k]) or one layer in [0, L)
 *          (cand_dev [B][k]); -1 entries pad a row.
 *   hits_dev / misses_dev: the counts ([B][L] or [B]), or NULL to discard
 *          them; misses are the rows the prefetch moved.
 * The slot tensor goes to scratch owned by the context, so calls on one
 * context must be ordered (as for every call).  Errors as skv_assemble;
 * captures into a CUDA graph. */
SKV_API skv_status skv_prefetch(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, int32_t layer,
                                const int32_t *cand_dev, int32_t *hits_dev, int32_t *misses_dev, skv_stream_t stream);

/* skv_prefetch with a built-in predictor, the recency window: the candidates
 * of request req_ids_dev[b] are its n newest tokens, [len - n, len) (all of
 * [0, len) when len < n), for every layer of the call, with len read on the
 * device when the call runs (after earlier write backs and extends on the
 * stream).  Decode-time Top-k favours recent tokens; keeping the window
 * resident turns those picks into hits.  0 <= n <= k, else
 * SKV_ERR_INVALID_ARG.  Candidates go to scratch owned by the context. */
SKV_API skv_status skv_prefetch_recent(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, int32_t layer, int32_t n,
                                       int32_t *hits_dev, int32_t *misses_dev, skv_stream_t stream);

/* skv_assemble for callers whose per-step tensors live in host memory
 * (pinned or pageable): copies req_ids [B] and topk [B][L][k] to device
 * staging buffers owned by the context, runs skv_assemble, and synchronises
 * `stream`.  An output (slots, hits, misses) in pinned host memory that the
 * device can address (cudaHostAlloc memory, torch's pin_memory) is written
 * by the kernels directly, over the host link in the direction the gather
 * does not use; any other output goes through a device staging buffer and a
 * copy back.  Same semantics and errors. */
SKV_API skv_status skv_assemble_host(skv_ctx *ctx, const int32_t *req_ids, int32_t B, const int32_t *topk, int32_t *slots,
                             int32_t *hits, int32_t *misses, skv_stream_t stream);

/* skv_assemble for callers that cannot allocate device memory when they
 * call: engines that reserve almost all HBM for their own pools at start-up
 * and allow no later cudaMalloc, or code that runs inside another
 * component's stream capture.  It allocates nothing and takes nothing from
 * the context's scratch: the gather work list lives in a file-scope static
 * device array of 2^20 (pool row, hot row) entries (8 MiB), which every
 * device that loads the library holds until the process exits.  Same
 * arguments, semantics and results as skv_assemble, except:
 *   - B * L * k must be <= 2^20, else SKV_ERR_INVALID_ARG (with the reason in
 *     skv_last_cuda_error) and nothing is enqueued;
 *   - skv_create loads the array on the context's device and looks up its
 *     address, so no call of this entry point loads or allocates anything;
 *   - every call on a device shares the one array: calls that overlap on the
 *     GPU (other streams, other contexts) race.  Nothing in the array needs
 *     to start at zero; the step resets its own counter.
 * The pages describe no counterpart of this entry point. */
SKV_API skv_status skv_assemble_noalloc(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, const int32_t *topk_dev,
                                        int32_t *slots_dev, int32_t *hits_dev, int32_t *misses_dev,
                                        skv_stream_t stream);

/* Release a request (lifecycle step "release"): its slot becomes free, its
 * maps are reset and its hot rows zeroed (enqueued on `stream`).  A later
 * skv_publish may hand the same id out again.  SKV_ERR_BAD_REQUEST if req is
 * not an active request.
 * Source: [xm] section "与SGLang HiSparse的集成" (release). */
SKV_API skv_status skv_release(skv_ctx *ctx, int32_t req, skv_stream_t stream);

/* Sparse MLA decode attention over assembled slots (the "compute" of
 * select-then-compute: "SGLang и Tair представили иерархичную Sparse Attention
 * ...", paragraph 2; the consumer of the slot tensor the index-copy step emits,
 * "Sparse Attention-Driven KVCache Management for Domestic AI Supernodes",
 * agenda item 2).  For each unit (batch entry b, layer l) of the call -- all L
 * layers when layer == -1 (units ordered b*L + l), else only `layer` (units
 * ordered b) -- with r = req_ids_dev[b]:
 *   keys_j = hot row (r, l, slots[unit][j]) for j < k, masked where the slot
 *            is -1 (or outside [0, S));
 *   s_hj   = sm_scale * sum_{d<576} q[unit][h][d] * keys_j[d]   (h < 128 heads)
 *   out[unit][h][0..512) = sum_j softmax_j(s_h)_j * keys_j[0..512)
 *   lse[unit][h] = log sum_j exp(s_hj)   (-inf and zero output if all masked)
 * q_dev is [units][128][576] bf16, slots_dev [units][k] int32 (as emitted by
 * skv_assemble / skv_assemble_layer), out_dev [units][128][512] bf16, lse_dev
 * [units][128] fp32 (may be null); device memory, q / out 16-byte aligned;
 * sm_scale finite and > 0 (else SKV_ERR_INVALID_ARG).
 * Requires row_bytes == 1152 (576 bf16).  Runs on the tensor cores (tcgen05):
 * QK^T and PV in tensor memory, fp32 accumulation, P rounded to bf16; a
 * cluster of two CTAs per unit, each owning half of the score dims and half of
 * the value dims, with the partial scores summed through distributed shared
 * memory.
 * Reads the hot buffer, so order it after the assemble that filled the slots
 * and before the next assemble of the same layer.  A product that does not
 * complete within a bounded wait sets SKV_DEVERR_TIMEOUT. */
SKV_API skv_status skv_attend(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, int32_t layer, const void *q_dev,
                              const int32_t *slots_dev, void *out_dev, float *lse_dev, float sm_scale,
                              skv_stream_t stream);

/* Read the sticky device error word into *bits (SKV_DEVERR_* mask, 0 = none)
 * and clear it.  Synchronises `stream`.
 * Source: the pages are silent on invalid input; this library's reading is
 * that a call with a bad request id or a bad or repeated Top-k entry is
 * rejected whole, and that a graph-executable step ([talk] agenda item 2,
 * UniDex; [xm] CUDA Graph support) reports it through device memory. */
SKV_API skv_status skv_get_device_error(skv_ctx *ctx, int32_t *bits, skv_stream_t stream);

/* Device address of the hot buffer and the bytes between consecutive
 * (request, layer) units (S * row_bytes).  Either pointer may be null.
 * Source: [talk] agenda item 2 (the device cache and the index mapping that
 * the attention kernel reads through: slot s of (r, l) is the row at
 * base + ((r*L + l)*S + s) * row_bytes). */
SKV_API skv_status skv_hot_buffer(skv_ctx *ctx, void **base, int64_t *unit_stride_bytes);

/* Host address of the pool; row (r, l, t) is at
 * base + ((r*L + l)*T_max + t) * row_bytes.  The same memory is mapped for
 * the device.  The caller may write rows [0, T) of a request it has just
 * published with rows == null, before the first skv_assemble on it. */
SKV_API skv_status skv_pool_rows(skv_ctx *ctx, void **host_base);

/* Debug / parity: copy one request's state to host memory after synchronising
 * `stream`.  Any output pointer may be null.  slot2tok, ts, lru are [L][S]
 * (lru as int32 slot ids, least recently used first), tok2slot is
 * [L][T_max], *len the request's token count, *active 1 or 0.
 * Source: [talk] agenda item 2 (the index mapping it exports); the pages
 * describe no export: it exists so the state can be checked. */
SKV_API skv_status skv_export_state(skv_ctx *ctx, int32_t req, int32_t *slot2tok, uint32_t *ts, int32_t *tok2slot,
                            int32_t *lru, int64_t *len, int32_t *active, skv_stream_t stream);

/* Debug / parity: copy one request's hot rows [L][S][row_bytes] to host
 * memory after synchronising `stream`. */
SKV_API skv_status skv_export_hot(skv_ctx *ctx, int32_t req, void *host_dst, skv_stream_t stream);

/* The step clock (number of successful skv_assemble calls), after
 * synchronising `stream`. */
SKV_API skv_status skv_get_clock(skv_ctx *ctx, uint32_t *clock, skv_stream_t stream);

/* Running totals since create, after synchronising `stream`: successful
 * assemble calls, hit entries and missed (gathered) rows. */
SKV_API skv_status skv_get_stats(skv_ctx *ctx, uint64_t *calls, uint64_t *hits, uint64_t *misses, skv_stream_t stream);

/* Where skv_create put the host pool.  On a host with several memory nodes
 * (a tray with two Grace CPUs, each linked to its own GPUs) a pool on the far
 * node would make every gather cross the CPU-to-CPU link as well, so
 * skv_create allocates the pool under a "preferred node" memory policy for the
 * host node nearest the context's GPU (skv_host_node_for_pci on "/sys"; the
 * environment variable SKV_POOL_NODE overrides it: a node id, or -1 for no
 * preference) and restores the caller's policy afterwards.
 *   *wanted_node  the node asked for, -1 if none;
 *   *seen_node    the node holding most of a sample of 64 pool pages as the
 *                 kernel reports them (move_pages), -1 if it reports none;
 *   *seen_frac    the share of that sample on *seen_node.
 * Any output pointer may be null.
 * Source: the pages are silent on host memory placement; the four decode GPUs
 * of [xm] section "XM-Sparse测试平台与解码性能" each serve their own batch,
 * which on a multi-socket host means one pool per GPU, each near its GPU. */
SKV_API skv_status skv_pool_placement(skv_ctx *ctx, int32_t *wanted_node, int32_t *seen_node, float *seen_frac);

/* The host NUMA node nearest a PCI device, read from a sysfs tree (host
 * code only; needs no GPU): the node whose CPU list shares the most CPUs with
 * the device's local_cpulist (lowest id on a tie); without a local CPU list,
 * the device's numa_node if that node has CPUs (a node without CPUs may be
 * GPU memory); else -1.  sysfs_root: null for "/sys" (a test passes a fake
 * tree); pci_bus_id as cudaDeviceGetPCIBusId prints it ("0000:01:00.0" or
 * with an 8-digit domain).  SKV_ERR_INVALID_ARG for null id or output. */
SKV_API skv_status skv_host_node_for_pci(const char *sysfs_root, const char *pci_bus_id, int32_t *node);

/* Optional timing hooks: when set (non-null), skv_assemble and
 * skv_assemble_layer record `before` just before the call's first kernel
 * (validation) and `after` just after the kernel that moves the missing rows
 * (the fused plan + gather kernel, which starts while validation runs), on
 * the call's stream (external event records, so they also work inside a
 * captured graph).  No event goes between the two kernels: it would keep them
 * from overlapping.  Pass two nulls to clear; passing exactly one null is
 * SKV_ERR_INVALID_ARG.  The events belong to the caller. */
SKV_API skv_status skv_set_gather_events(skv_ctx *ctx, skv_event_t before, skv_event_t after);

/* Optional: the attention kernel of later skv_attend calls on this context
 * occupies at most `sms` SMs (one CTA per SM, in clusters of two; rounded
 * down to an even count, at least 2), leaving the others to work running at
 * the same time on other streams -- e.g. the next layer's skv_assemble_layer,
 * which is bound by the host link and needs few SMs to keep it busy.  0 (the
 * default) uses every SM.  Negative: SKV_ERR_INVALID_ARG.  Results do not
 * depend on it. */
SKV_API skv_status skv_set_attend_sms(skv_ctx *ctx, int32_t sms);

/* Diagnostic: one 128 x n x k bf16 matrix product on the tensor cores through
 * the same path the attention consumer uses (tcgen05 MMA into tensor memory,
 * read back by the issuing warpgroup):
 * d_dev[128][n] (fp32) = a_dev[128][k] * B^T.  `mode` bit 0 clear: B = b_dev
 * as [n][k] row-major, staged K-major; set: B^T = b_dev as [k][n] row-major,
 * staged MN-major (the form in which the attention consumer reads V).  Bit 1
 * clear: A staged K-major in shared memory; set: A written to tensor memory
 * (row m in lane m, two bf16 per 32-bit column) and read from there (the form
 * in which the attention consumer holds Q).  Device memory, a / b 16-byte
 * aligned, 16 <= n <= 256 and 16 <= k <= 128, both multiples of 16,
 * 0 <= mode <= 3, else SKV_ERR_INVALID_ARG.  Allocates a 4-byte status word
 * with cudaMallocAsync and synchronises `stream`.  SKV_ERR_CUDA (with a
 * message) if the MMA does not complete within a bounded wait.  Not part of
 * any decode step. */
SKV_API skv_status skv_selftest_mma(const void *a_dev, const void *b_dev, float *d_dev, int32_t n, int32_t k,
                                    int32_t mode, skv_stream_t stream);

/* Diagnostic of skv_attend's bounded waits (not part of any decode step):
 * launches the attention kernel over the call's units (all layers; arguments
 * as skv_attend, out_dev [units][128][512] bf16) exactly as skv_attend would,
 * except that the kernel never issues a key load.  Its first wait for keys
 * therefore runs out (within about two seconds) with no copy and no
 * tensor-core product in flight; the kernel sets SKV_DEVERR_TIMEOUT in the
 * sticky error word and winds down, leaving out_dev unspecified.  Lets a test
 * show that a wait that runs out ends in an error status the host can read
 * (skv_get_device_error) and that the context stays usable, without faulting
 * or hanging a GPU.  Host errors as skv_attend. */
SKV_API skv_status skv_selftest_attend_timeout(skv_ctx *ctx, const int32_t *req_ids_dev, int32_t B, const void *q_dev,
                                               const int32_t *slots_dev, void *out_dev, skv_stream_t stream);

/* The message of the last failing CUDA call on this thread ("" if none). */
SKV_API const char *skv_last_cuda_error(void);

/* Human-readable name of a status. */
SKV_API const char *skv_status_string(skv_status s);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H_ */
