/*
 * lora.h - C boundary of the GB300 multi-adapter LoRA projection library (liblora.so).
 *
 * What it computes ("S-LoRA, in depth", section "Merge or keep adapters separate"):
 * for a batch of T tokens, each carrying its own adapter id a(t), one projection
 * slot computes
 *
 *     y_t = x_t W + (x_t A_{a(t)}) B_{a(t)}          (unmerged LoRA)
 *
 * with W shared by every token (H x H) and the low-rank factors A (H x r),
 * B (r x H) of the token's own adapter, r in [1, 64].  A token with adapter id -1
 * gets y_t = x_t W.  The factors live in a unified page pool (same page, section
 * "Unified paging: adapters and KV cache in one pool"): the pool is an array of
 * pages, one page holds one vector of H values, a rank-r A or B takes r pages, and
 * adapter pages come from the same free list as KV-cache pages.
 *
 * Conventions for every entry point
 *  - Pointers named *_host are host memory; every other data pointer is device memory
 *    on the current CUDA device.  Device memory for x, W, y, the pool storage and the
 *    segment workspace is owned by the caller (e.g. PyTorch tensors); the library keeps
 *    non-owning pointers and never frees them.
 *  - Element types: bf16 for pool pages, x, W, y and the host A/B factors (raw 16-bit
 *    patterns); fp32 for the optional LoRA delta; int32 for token adapter ids.
 *  - Device work is enqueued on the caller's stream (a cudaStream_t passed as
 *    lora_stream_t; NULL = the legacy default stream).  Only lora_adapter_load (also when
 *    lora_adapter_ensure loads) and lora_status synchronise that stream.
 *  - Return value: LORA_OK (0) or a negative LORA_E* code; lora_last_error() then gives
 *    a message for the calling thread.  A failing call leaves the pool as it was (one
 *    exception, stated at lora_adapter_ensure: a load that fails with LORA_ECUDA after
 *    idle adapters were evicted for it keeps those evictions).
 *  - Adapters are immutable once loaded; there is no global "active adapter": the
 *    adapter of every token travels in each call ("Switch Adapters by Routing Requests
 *    Through Resident, Verified State": request-scoped binding; an unknown adapter is
 *    an error).
 *  - One pool may be used from one host thread at a time.
 */
#ifndef ADAPTER_GEMM_LORA_H
#define ADAPTER_GEMM_LORA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lora_stream_t;  /* identical to cudaStream_t */

#define LORA_OK                0
#define LORA_EINVAL           -1   /* null pointer, bad size, H % 64 != 0, slot or id out of range */
#define LORA_ENOPAGES         -2   /* the free list holds fewer pages than asked for */
#define LORA_EUNKNOWN_ADAPTER -3   /* adapter id not loaded */
#define LORA_ERANK            -4   /* rank outside [1, LORA_MAX_RANK] */
#define LORA_EEXIST           -5   /* adapter id already loaded */
#define LORA_ECUDA            -6   /* a CUDA runtime or driver call failed */
#define LORA_EDEVICE          -7   /* a device-side check failed (see lora_status) */
#define LORA_EBUSY            -8   /* the adapter has active requests */

#define LORA_MAX_RANK      64
#define LORA_MAX_ADAPTERS  16384    /* adapter ids are indices in [0, max_adapters) */
#define LORA_MAX_TOKENS    65536    /* tokens per batch */
#define LORA_MAX_GROUP     4        /* slots per lora_linear_forward_group call */

typedef struct lora_pool lora_pool;

typedef struct lora_pool_stats_t {
  int64_t num_pages;
  int64_t free_pages;
  int64_t adapter_pages;
  int64_t reserved_pages;      /* KV / filler pages: lora_pool_reserve and lora_kv_grow */
  int32_t resident_adapters;
  int32_t max_adapters;
} lora_pool_stats_t;

/*
 * Per-batch token grouping, built on the device by lora_segments_build and read by
 * lora_linear_forward.  Set up with lora_segments_init over a caller-allocated device
 * workspace of lora_segments_size() bytes; every pointer below points into it.
 * Device arrays (after a build with T tokens, S = *n_seg segments):
 *   perm[T]          token indices, stable-sorted by adapter id; id -1 tokens first;
 *   seg_off[S + 1]   segment s covers perm[seg_off[s] .. seg_off[s+1]); seg_off[0] is
 *                    the number of no-adapter tokens and seg_off[S] = T;
 *   seg_adapter[S]   adapter id of segment s, ascending;
 *   n_seg[1]         S;
 *   units[4 U]       LoRA-delta work units, U = *n_units: unit u covers the tokens
 *                    perm[units[4u+2] .. units[4u+2] + units[4u+3]) (at most 16, all of one
 *                    segment) of adapter units[4u], whose rank is units[4u+1]; listed by
 *                    rank class (33..64, 17..32, 9..16, 1..8), then adapter id, then offset;
 * plus the fp32 scratch for the LoRA delta used by lora_linear_forward (delta_slots
 * buffers of [T_max][H], one per slot of a lora_linear_forward_group call).  Calls that use
 * the same workspace must be ordered on one stream: the scratch is reused by every
 * projection slot.
 */
typedef struct lora_segments {
  int32_t T_max;          /* token capacity of the workspace */
  int32_t T;              /* tokens of the last build (host copy), -1 before any build */
  int32_t max_seg;        /* capacity of the segment arrays */
  int32_t H;              /* hidden size of the pool the workspace was sized for */
  int32_t* perm;
  int32_t* seg_off;
  int32_t* seg_adapter;
  int32_t* n_seg;
  int32_t* tok_adapter;   /* [T_max] validated adapter id per token (-1 = none or rejected) */
  int32_t* units;         /* [4 * unit_cap] (adapter, rank, first perm index, tokens) */
  int32_t* n_units;
  int32_t unit_cap;
  int32_t delta_slots;    /* fp32 delta buffers at `delta` (the workspace's max_group) */
  float*   delta;         /* [delta_slots][T_max][H]  (x_t A) B (fp32) */
  float*   gemm_partials; /* [delta_slots][3][P][H] fp32 partial sums of the base GEMM for batches
                             of <= 256 tokens (K split over 4 CTAs); P = min(T_max, 256) rounded
                             up to 128 */
  /* Batches of more than 256 tokens (prefill-shaped; empty when T_max <= 256): the batch is cut
   * into tiles of 256 consecutive tokens, and a tile whose tokens carry at most
   * LORA_TILE_ADAPTERS distinct adapters ("a fused tile") gets its LoRA term inside the base
   * GEMM (see lora_linear_forward).  After a build: */
  int32_t  n_tiles_max;   /* capacity: T_max / 256 rounded up (0 when T_max <= 256) */
  int32_t* tile_plan;     /* [n_tiles_max][8]: [0] = adapters of tile i, or -1 when it has more than
                             LORA_TILE_ADAPTERS; [1..4] their ids, ascending */
  int32_t* entries;       /* [4 * n_tiles_max]: the fused (tile, adapter slot b) pairs, tile * 4 + b,
                             in tile order */
  int32_t* n_entries;
  int32_t* units_rest;    /* [4 * unit_cap]: the work units (records as in units) that hold at
                             least one token of a non-fused tile, in the order of units; the token
                             count of a unit that also holds tokens of fused tiles has bit 8 (256)
                             set */
  int32_t* n_units_rest;
  uint16_t* s_lora;       /* [delta_slots][T_max][512] bf16: per token of a fused tile, s = x A of
                             its adapter as hi and lo bf16 parts in the columns of its tile slot */
  float*   shrink_scratch;/* fp32 partial sums exchanged by the shrink kernel's CTAs */
} lora_segments;

#define LORA_TILE_TOKENS   256      /* tokens per tile of a prefill-shaped batch */
#define LORA_TILE_ADAPTERS 4        /* distinct adapters a fused tile may carry */

/*
 * Create a pool over caller-owned device storage.
 *   pool_dev         device bf16 [num_pages][H]; NULL creates a planning pool that only
 *                    does the page bookkeeping (no device memory, no copies, no kernels);
 *   num_pages        1 .. 2^31-1;   H: multiple of 64, 64 .. 16384;
 *   n_slots          projection slots (e.g. 4 per layer for q, k, v, o), >= 1;
 *   max_adapters     adapter ids must lie in [0, max_adapters), 1 .. LORA_MAX_ADAPTERS;
 *   page_order_host  nullable int64 [num_pages]: the initial free list (a permutation of
 *                    0..num_pages-1); pages are taken from its END, as the pool sketch in
 *                    "Unified paging" pops its free list.  NULL = 0, 1, ..., num_pages-1.
 * The library allocates its own device page tables (max_adapters * n_slots * 512 bytes)
 * and an error word.  *out receives the handle; free it with lora_pool_destroy.
 */
int lora_pool_create(void* pool_dev, int64_t num_pages, int32_t H, int32_t n_slots,
                     int32_t max_adapters, const int64_t* page_order_host, lora_pool** out);

/* Take n pages from the free list for KV cache or other non-adapter use (the sketch's
 * grow_kv).  page_ids_host (int64 [n], out) receives them in the order taken.
 * LORA_ENOPAGES if fewer than n are free (nothing taken). */
int lora_pool_reserve(lora_pool* pool, int64_t n, int64_t* page_ids_host);

/*
 * KV-cache pages of a request ("Unified paging": a sequence of length S takes S pages per K and
 * per V; the pool sketch's grow_kv takes 2 * layers pages for each new token, from the same free
 * list as adapter pages).
 *   lora_kv_grow: n_tokens new tokens of `request_id` (any int64 key); each takes 2 * layers
 *     pages from the end of the free list, per layer ascending its K page then its V page.
 *     page_ids_host (nullable, out: int32 [n_tokens * 2 * layers]) receives them in that order.
 *     LORA_ENOPAGES if fewer are free (nothing taken: the caller preempts or aborts, as in the
 *     sketch); LORA_EINVAL for n_tokens < 0, layers < 1, or a layer count that differs from the
 *     request's first growth.
 *   lora_kv_free: a finished request gives every KV page back, in the order taken
 *     (LORA_EINVAL if the request holds none).
 *   lora_kv_length: the request's cached tokens, or -1 if it holds no pages.
 *   lora_kv_table: table_host (out: int32 [tokens][2]) = (K page, V page) of every cached token
 *     at `layer`, in token order.
 * These are host bookkeeping; they count as reserved pages in lora_pool_stats and cannot be
 * given back through lora_pool_release.
 */
int lora_kv_grow(lora_pool* pool, int64_t request_id, int32_t n_tokens, int32_t layers, int32_t* page_ids_host);
int lora_kv_free(lora_pool* pool, int64_t request_id);
int64_t lora_kv_length(const lora_pool* pool, int64_t request_id);
int lora_kv_table(const lora_pool* pool, int64_t request_id, int32_t layer, int32_t* table_host);

/*
 * Decode attention over KV pages of the pool ("Unified paging": a token's K and V at each layer
 * are one page each, so adapter pages and KV pages share one pool and one free list).  For one
 * new token per request, at `layer`, per head h of width D = H / n_heads (D = 64 or 128):
 *     out_h = softmax_j( q_h . K_{j,h} / sqrt(D) ) V_{j,h}      over the request's cached tokens j
 * (plain scaled dot-product attention; the pages give no formula of their own).
 *   lora_kv_batch_table: writes table_dev (device int32 [n_req][max_len][layers][2]: every
 *     request's KV page list as lora_kv_grow took it, -1 past its length) and seq_len_dev
 *     (device int32 [n_req]); every request must hold pages, with one layer count, and at most
 *     max_len tokens (LORA_EINVAL otherwise).  Synchronises `stream` (its host staging is reused).
 *   lora_attention_decode: q and out device bf16 [n_req][H] (16-byte aligned); out is rounded
 *     to bf16 once from fp32.  A request with no cached token gets zeros.  Page ids outside the
 *     pool set the device error word (lora_status) and their tokens are skipped.  One kernel;
 *     at most 65535 requests per call.
 */
int lora_kv_batch_table(lora_pool* pool, const int64_t* request_ids_host, int32_t n_req, int32_t max_len,
                        int32_t* table_dev, int32_t* seq_len_dev, lora_stream_t stream);
int lora_attention_decode(lora_pool* pool, int32_t n_req, const int32_t* table_dev, const int32_t* seq_len_dev,
                          int32_t max_len, int32_t layers, int32_t layer, const void* q, void* out, int32_t n_heads,
                          lora_stream_t stream);

/* Give back n reserved pages (appended to the free list in the order given).
 * LORA_EINVAL if any id is not currently reserved or appears twice (nothing released). */
int lora_pool_release(lora_pool* pool, int64_t n, const int64_t* page_ids_host);

/*
 * Load an adapter ("Unified paging" sketch, ensure_adapter): take 2 * rank pages per slot
 * that carries LoRA and copy the factors into them.
 *   A_host[slot]   host bf16 [H][rank] row-major, or NULL: no LoRA on that slot;
 *   B_host[slot]   host bf16 [rank][H] row-major (ignored where A_host[slot] is NULL);
 *   page_table_host (out, nullable) int32 [n_slots][2][rank]: [slot][0][j] = page holding
 *                  column j of A, [slot][1][j] = page holding row j of B, -1 for a slot
 *                  without LoRA.  Pages are taken in that order (slot, A then B, j).
 * In a planning pool A_host may be NULL (every slot carries LoRA) and no data is read.
 * Synchronises `stream` (the host staging buffer is reused).
 * Errors: LORA_EINVAL (id range, null B where A is set), LORA_ERANK, LORA_EEXIST,
 * LORA_ENOPAGES (pool unchanged), LORA_ECUDA.
 */
int lora_adapter_load(lora_pool* pool, int32_t adapter_id, int32_t rank,
                      const void* const* A_host, const void* const* B_host,
                      lora_stream_t stream, int32_t* page_table_host);

/*
 * Loads that overlap compute ("S-LoRA, in depth", "Scheduling": the prefetcher copies the next
 * batch's adapters while the current batch computes; pinned host memory and a separate copy
 * stream make the overlap possible).  An adapter is packed once, on the host, into page rows in
 * the order lora_adapter_load takes pages (slot, A columns then B rows, j ascending), behind a
 * header the load fills in; the caller keeps the packed form in pinned (page-locked) host memory.
 *   lora_adapter_packed_size: bytes of the packed form for `rank` on the slots marked in
 *     present_host (nullable int32 [n_slots], non-zero = LoRA on that slot; NULL = every slot).
 *   lora_adapter_pack: host only; A_host / B_host as for lora_adapter_load (NULL A = no LoRA
 *     on that slot, which must agree with present_host at load time).
 *   lora_adapter_load_packed: takes the adapter's pages at once (host bookkeeping, same order
 *     and errors as lora_adapter_load) and enqueues on `copy_stream` one kernel that reads the
 *     packed rows straight from the pinned buffer into those pages and writes the adapter's
 *     device page table and rank; it does not synchronise.  Before reusing pages it makes
 *     copy_stream wait for the last unload or eviction, so batches enqueued before that still
 *     read the old contents.  The buffer must be pinned host memory (LORA_EINVAL otherwise),
 *     16-byte aligned, and unchanged until copy_stream has passed the load.
 *   lora_adapter_wait: makes `stream` wait for the adapter's last packed load (no-op after a
 *     synchronous load); work on `stream` that uses the adapter must come after it.
 * Unload and eviction of an adapter whose packed load may be in flight wait for it first.
 */
int64_t lora_adapter_packed_size(const lora_pool* pool, int32_t rank, const int32_t* present_host);
int lora_adapter_pack(const lora_pool* pool, int32_t rank, const void* const* A_host, const void* const* B_host,
                      void* packed_host, int64_t packed_bytes);
int lora_adapter_load_packed(lora_pool* pool, int32_t adapter_id, int32_t rank, const int32_t* present_host,
                             const void* packed_pinned, int64_t packed_bytes, lora_stream_t copy_stream,
                             int32_t* page_table_host);
int lora_adapter_wait(lora_pool* pool, int32_t adapter_id, lora_stream_t stream);

/* Return an adapter's pages to the free list (in the order they were taken) and clear its
 * device page table (enqueued on `stream`; work already enqueued before it on that stream
 * still sees the adapter).  LORA_EUNKNOWN_ADAPTER if it is not loaded, LORA_EBUSY if it has
 * active requests (see lora_adapter_acquire). */
int lora_adapter_unload(lora_pool* pool, int32_t adapter_id, lora_stream_t stream);

/* Device workspace bytes lora_segments_init needs for batches of up to T_max tokens
 * (dominated by the fp32 delta, T_max * H * 4 bytes).  Returns < 0 on bad arguments. */
int64_t lora_segments_size(const lora_pool* pool, int32_t T_max);

/* Carve `workspace_dev` (>= lora_segments_size bytes, 256-byte aligned) into *seg. */
int lora_segments_init(const lora_pool* pool, void* workspace_dev, int64_t workspace_bytes,
                       int32_t T_max, lora_segments* seg);

/* The same for a workspace that also serves lora_linear_forward_group calls of up to
 * max_group (1 .. LORA_MAX_GROUP) slots: it holds max_group delta buffers and max_group
 * split-K scratch areas instead of one.  lora_segments_size/init are these with max_group = 1. */
int64_t lora_segments_size_group(const lora_pool* pool, int32_t T_max, int32_t max_group);
int lora_segments_init_group(const lora_pool* pool, void* workspace_dev, int64_t workspace_bytes,
                             int32_t T_max, int32_t max_group, lora_segments* seg);

/*
 * Group a batch's tokens by adapter (stable: ascending adapter id, ties by token index).
 *   token_adapter  device int32 [T]: adapter id per token, -1 = no adapter;
 *   T              0 .. seg->T_max.
 * Ids that are not loaded are treated as "no adapter" and raise the device error word
 * (LORA_EUNKNOWN_ADAPTER, reported by lora_status).  Built once per batch, reused by every
 * slot's lora_linear_forward.
 */
int lora_segments_build(lora_pool* pool, const int32_t* token_adapter, int32_t T,
                        lora_segments* seg, lora_stream_t stream);

/*
 * One projection slot over the batch last built into `seg`:
 *     y[t, n] = bf16_rne( sum_k x[t,k] W[n,k]  +  sum_j s[t,j] B_{a(t)}[j, n] ),
 *     s[t, j] = sum_k x[t,k] A_{a(t)}[k, j]        (fp32; bf16 inputs, fp32 accumulation)
 *   x      device bf16 [T][H] row-major;
 *   W      device bf16 [H][H] in nn.Linear layout W[out][in] (so y = x W^T);
 *   y      device bf16 [T][H] row-major, written (out of place; must not alias x);
 *   delta_dbg  nullable device fp32 [T][H]: receives the LoRA term alone (0 for tokens
 *          without LoRA on this slot), for parity tests.
 * Kernels: the LoRA delta (paged shrink and expand fused, s kept on chip), then the tcgen05
 * base GEMM with an epilogue that adds the delta before the single bf16 rounding.
 * Errors: LORA_EINVAL (slot, pointers, no batch built), LORA_ECUDA (launch failure).
 */
int lora_linear_forward(lora_pool* pool, const lora_segments* seg, int32_t slot,
                        const void* x, const void* W, void* y, float* delta_dbg,
                        lora_stream_t stream);

/*
 * n projection slots that read the same input x, e.g. the q, k and v projections of one layer
 * ("S-LoRA, in depth", "The architecture": every layer's projections run over the whole
 * batch; q, k and v all take the layer's hidden state).  Computes, for each i < n, exactly
 * what lora_linear_forward(pool, seg, slots_host[i], x, W_host[i], y_host[i],
 * delta_dbg_host[i], stream) computes, bit for bit, but the LoRA deltas of all n slots come
 * from one kernel launch (its work list is every unit of the batch once per slot), followed
 * by the n base GEMMs.
 *   n               1 .. seg->delta_slots (see lora_segments_init_group);
 *   slots_host      host int32 [n], distinct slots;
 *   W_host, y_host  host arrays [n] of device pointers (W[out][in] bf16, y bf16 [T][H]); no y
 *                   may alias x or another y;
 *   delta_dbg_host  nullable host array [n] of nullable device fp32 [T][H] pointers.
 * Errors: as lora_linear_forward; LORA_EINVAL also for n outside 1 .. seg->delta_slots or
 * a repeated slot.
 */
int lora_linear_forward_group(lora_pool* pool, const lora_segments* seg, int32_t n, const int32_t* slots_host,
                              const void* x, const void* const* W_host, void* const* y_host,
                              float* const* delta_dbg_host, lora_stream_t stream);

/*
 * Adapter lifecycle in the unified pool ("S-LoRA, in depth", "Unified paging": the pool sketch
 * counts each resident adapter's active requests; ensure_adapter loads an adapter that is not
 * resident, first evicting idle adapters, those with no active request, to free pages; "The
 * architecture": when an adapter has no active requests left, its pages can be reclaimed for
 * KV cache or for another adapter).
 *   lora_adapter_load leaves a new adapter resident and idle (0 active requests);
 *   lora_adapter_acquire / lora_adapter_release add / remove one active request
 *     (LORA_EUNKNOWN_ADAPTER if not resident; release of an idle adapter is LORA_EINVAL);
 *   lora_adapter_refs returns the count, or -1 if the adapter is not resident;
 *   lora_adapter_unload refuses an adapter with active requests (LORA_EBUSY).
 */
int lora_adapter_acquire(lora_pool* pool, int32_t adapter_id);
int lora_adapter_release(lora_pool* pool, int32_t adapter_id);
int32_t lora_adapter_refs(const lora_pool* pool, int32_t adapter_id);

/*
 * Which idle adapter is evicted first ("Fewer Expert Transfers Without Changing Routing",
 * sections "A better eviction rule cuts transfers without changing routing" and "Limited
 * foresight": an eviction choice changes only future loads, never the current batch's work):
 *   LORA_EVICT_LOAD_ORDER  the one loaded earliest (the pool sketch; the default);
 *   LORA_EVICT_LRU         the least recently used (last load, ensure or acquire);
 *   LORA_EVICT_FARTHEST    the one whose next request in `future_host` lies farthest; only the
 *                          first `lookahead` entries are looked at (<= 0: all of them), and the
 *                          adapters not requested there count as equal and go first, least
 *                          recently used first.
 * future_host (nullable when n_future is 0) is copied; callers refresh it as their queue moves.
 * LORA_EINVAL for an unknown policy or n_future < 0.
 */
#define LORA_EVICT_LOAD_ORDER 0
#define LORA_EVICT_LRU        1
#define LORA_EVICT_FARTHEST   2
int lora_pool_set_eviction(lora_pool* pool, int32_t policy, const int32_t* future_host, int64_t n_future,
                           int32_t lookahead);

/*
 * Evict idle adapters, in the order of the pool's eviction rule (lora_pool_set_eviction; by
 * default the one loaded earliest first), until at least `need` pages are free (the sketch's
 * evict_idle_adapters), clearing their device page tables in `stream` order as
 * lora_adapter_unload does: work enqueued on `stream` before the call still sees them.
 *   evicted_host  nullable host int32 [max_adapters]: receives the evicted ids in order;
 *   n_evicted     nullable: receives their count.
 * If evicting every idle adapter would still leave fewer than `need` pages free, nothing is
 * evicted and the call returns LORA_ENOPAGES (the sketch evicts them and still fails).
 */
int lora_pool_evict_idle(lora_pool* pool, int64_t need, lora_stream_t stream, int32_t* evicted_host,
                         int32_t* n_evicted);

/*
 * The sketch's ensure_adapter.  If `adapter_id` is resident it gets one more active request
 * (A_host and B_host are not read; `rank` must equal the resident rank, else LORA_ERANK) and
 * *loaded_out = 0.  Otherwise idle adapters are evicted as lora_pool_evict_idle does to make
 * room for its pages, the adapter is loaded as lora_adapter_load does (same arguments, same
 * page order) and given one active request, and *loaded_out = 1.  table_out as for
 * lora_adapter_load; evicted_host / n_evicted as for lora_pool_evict_idle (all nullable).
 * LORA_ENOPAGES (nothing evicted, nothing loaded) if even evicting every idle adapter would
 * not free enough pages; argument errors are found before anything is evicted.  If the load
 * itself then fails with LORA_ECUDA, the evictions made for it stand.
 */
int lora_adapter_ensure(lora_pool* pool, int32_t adapter_id, int32_t rank, const void* const* A_host,
                        const void* const* B_host, lora_stream_t stream, int32_t* table_out,
                        int32_t* loaded_out, int32_t* evicted_host, int32_t* n_evicted);

/* Synchronise `stream`, read and clear the device error word.  LORA_OK, or LORA_EDEVICE
 * with lora_last_error() naming the failed check (unknown adapter id, page id out of
 * range, bad rank, a bounded wait that ran out). */
int lora_status(lora_pool* pool, lora_stream_t stream);

/* Page accounting: free, adapter and reserved pages, resident adapters. */
void lora_pool_stats(const lora_pool* pool, lora_pool_stats_t* out);

/* Message for the last non-zero status returned on the calling thread ("" if none). */
const char* lora_last_error(void);

/*
 * Kernel accounting for benchmarks.  Every kernel this library launches for `pool` is counted
 * by kind: 0 segment build, 1 LoRA delta (shrink and expand), 2 base GEMM, 3 page scatter
 * (adapter loads), 4 shrink of the fused tiles of a prefill-shaped batch, 5 decode attention.
 * With profiling enabled, each launch is also bracketed by CUDA events recorded on the
 * stream it runs on (also inside a stream capture: the events then become graph nodes and
 * are re-recorded by every replay).  lora_profile_read synchronises those events and
 * writes, for kinds 0 .. n_kinds-1, the launch count and the summed device milliseconds
 * (0 where profiling was off); with `reset` != 0 it then clears both records.
 * Events cost ~1 us of host time per launch.
 */
#define LORA_KIND_SEGMENTS 0
#define LORA_KIND_DELTA    1
#define LORA_KIND_GEMM     2
#define LORA_KIND_SCATTER  3
#define LORA_KIND_SHRINK   4
#define LORA_KIND_ATTENTION 5
#define LORA_N_KINDS       6
int lora_profile_enable(lora_pool* pool, int32_t enable);
int lora_profile_read(lora_pool* pool, int32_t n_kinds, int64_t* launches_host, double* ms_host,
                      int32_t reset);

/*
 * lora_linear_forward_noalloc: the same projection as lora_segments_build followed by
 * lora_linear_forward, for callers that cannot allocate device memory (no counterpart on the
 * pages; it exists for library users).  Examples: a plugin whose host runtime owns all device
 * memory and passes it only inputs and outputs; code recording a CUDA graph while stream
 * capture forbids cudaMalloc; a latency-critical loop that must not risk the device-wide
 * synchronisation an allocation can bring.  The segment data and fp32 scratch live in one
 * static device array of LORA_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits; nothing is allocated per call.
 *   token_adapter  device int32 [T], -1 = no adapter;  T in 0 .. LORA_NOALLOC_MAX_TOKENS;
 *   x, W, y        as for lora_linear_forward;  pool H must not exceed LORA_NOALLOC_MAX_H.
 * The first call on each device looks the array's device address up (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.  All calls share
 * the array: calls whose work overlaps on the GPU (several streams or host threads) race,
 * calls ordered on one stream do not.  No value in it needs to start at zero.
 * Errors: LORA_EINVAL for T or H above the limits (message names the limit) and as for
 * lora_linear_forward; LORA_ECUDA.
 */
#define LORA_NOALLOC_MAX_TOKENS 128
#define LORA_NOALLOC_MAX_H 8192
#define LORA_NOALLOC_SCRATCH_BYTES (17 * 1024 * 1024)
int lora_linear_forward_noalloc(lora_pool* pool, const int32_t* token_adapter, int32_t T, int32_t slot,
                                const void* x, const void* W, void* y, lora_stream_t stream);

/* Free the pool's own host and device memory (not the caller's storage). NULL is ignored. */
void lora_pool_destroy(lora_pool* pool);

#ifdef __cplusplus
}
#endif

#endif /* ADAPTER_GEMM_LORA_H */
