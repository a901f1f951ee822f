/*
 * sglattn.h -- C ABI of the GB300 RadixAttention hot path (libsglattn.so).
 *
 * What the library computes, and where the pages on SGLang define it:
 *
 *  - A host radix tree over a token-granular KV pool: longest-prefix match,
 *    insert with node split, per-request reference counts, leaf-first LRU
 *    eviction, and one free list shared by cache and running requests.
 *    ["SGLang 深度拆解" (chenxutan.com/d/5669.html) §2.3; bhfrc.com/news/45689
 *    §3.1-§3.2; "SGLang：从前端 DSL 到 SRT 服务运行时" (oripoin.cn), section
 *    "用基数树实现前缀复用"]
 *  - The batch tables RadixAttention reads: req_to_token (request -> token
 *    position -> pool slot) and the prefix groups (runs of positions that a
 *    set of requests shares), so a shared prefix is read once.
 *    ["SGLang 深度解读" (luoboask.github.io/fde-learning/opensource/sglang/),
 *    sections "1. RadixCache" and "5. Attention 层"; bhfrc.com §1.3]
 *  - Decode attention (one query token per request over its context) and
 *    extend attention (new tokens over a cached prefix plus a causal new
 *    block), returning O and the natural-log log-sum-exp per (row, head).
 *    ["SGLang 深度拆解" §3.2 (what its PagedDecode / PagedPrefill sketches
 *    compute) and §4.1 (decode is memory-bound, prefill compute-bound)]
 *
 * Conventions (all entry points):
 *  - Every function returns an int status: SGL_OK (0) or a negative
 *    SGL_ERR_* code.  sgl_status_string() names it.  A failed call leaves
 *    outputs unspecified unless its comment says otherwise.
 *  - The caller owns every array it passes.  The library owns sgl_tree,
 *    sgl_groups and sgl_plan objects; each has a destroy function.  Views
 *    returned by the library point into library memory and stay valid until
 *    the owning object is destroyed or refilled.
 *  - "host" pointers are ordinary CPU memory; "device" pointers are CUDA
 *    global memory of the current device.  GPU entry points are asynchronous
 *    on the given stream; host-detected errors return immediately, launch
 *    errors as SGL_ERR_CUDA (sgl_last_cuda_error() gives the cudaError_t),
 *    and data errors found by the kernels (a slot outside the pool, a plan
 *    that disagrees with seq_lens) as SGL_ERR_BOUNDS from sgl_check().
 *  - No entry point allocates device memory.  There is no CPU fallback: if
 *    the GPU path cannot run, the call fails.
 *  - Supported: head_dim 64 or 128; Hq / Hkv in {1, 2, 4, 8}; fp32 or bf16
 *    Q/K/V (one dtype for all three and for O).  Others: SGL_ERR_UNSUPPORTED.
 *  - Pool layout: K and V are two device buffers [num_slots, Hkv, head_dim]
 *    (slot-major; one slot holds one token of one layer).  With page_size P
 *    > 1, slot = page * P + offset and a page's P slots are contiguous.
 *  - Query head h reads KV head h / (Hq / Hkv).  sm_scale <= 0 means
 *    1 / sqrt(head_dim).
 */
#ifndef SGLATTN_H
#define SGLATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t-compatible opaque stream handle (NULL = legacy default stream). */
typedef struct CUstream_st* sgl_stream_t;

enum {
    SGL_OK = 0,
    SGL_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad handle, malformed input */
    SGL_ERR_NO_SLOTS = -2,    /* pool exhausted even after evicting every unreferenced leaf */
    SGL_ERR_UNSUPPORTED = -3, /* dtype / head_dim / group size outside the supported set */
    SGL_ERR_CUDA = -4,        /* a CUDA call failed; see sgl_last_cuda_error() */
    SGL_ERR_BOUNDS = -5,      /* a kernel met a slot or position outside its tables */
    SGL_ERR_STATE = -6,       /* unlock below zero, or a stale node handle */
    SGL_ERR_WORKSPACE = -7    /* workspace missing, misaligned or too small */
};

enum { SGL_DTYPE_F32 = 0, SGL_DTYPE_BF16 = 1, SGL_DTYPE_BF16_FP8KV = 2 };
/* SGL_DTYPE_BF16_FP8KV: Q and O bf16, the K and V pools FP8 E4M3 bytes
 * (decode and extend); K = k_scale * pool value, V = v_scale * pool value
 * (per-tensor scales in sgl_attn_params).  sgl_extend_attn_kvwrite takes
 * bf16 k_new / v_new and stores round-to-nearest-even E4M3 codes of
 * k_new / k_scale and v_new / v_scale (saturating at +-448, NaN kept).  The
 * query enters the tensor cores as f16: a query element outside the f16
 * range sets SGL_ERR_BOUNDS for sgl_check.  ["SGLang 深度拆解" (the FP8 KV
 * cache halves the KV bytes); CS349D lecture-16 notes §4 (FP8 KV cache)] */

/* Name of a status code (static string). */
const char* sgl_status_string(int status);
/* The cudaError_t of the last SGL_ERR_CUDA raised on this thread (0 if none). */
int sgl_last_cuda_error(void);
/* Library version string (static). */
const char* sgl_version(void);

/* ======================================================================== */
/* Host radix tree                                                          */
/* ======================================================================== */

typedef struct sgl_tree sgl_tree;
/* Node handle: 0 is the root; other handles stay valid while the node exists
 * (a node split keeps the handle on the lower part, which ends where the
 * node ended).  A handle of an evicted node gives SGL_ERR_STATE. */
typedef int64_t sgl_node;

/* Create a tree over a pool of num_slots slots in pages of page_size slots
 * (num_slots % page_size == 0).  free_order (host, num_slots / page_size
 * entries, a permutation of page ids) is the initial free list; NULL means
 * 0, 1, 2, ...  alloc pops pages from the front; freed and evicted pages are
 * appended to the back in the order they are released.
 * [oripoin.cn, "用基数树实现前缀复用": cache and running requests share one pool] */
int sgl_tree_create(int64_t num_slots, int32_t page_size, const int32_t* free_order, sgl_tree** out);
void sgl_tree_destroy(sgl_tree* tree);

/* Longest prefix of tokens[0..n) held by the tree, in whole pages.
 * Writes matched_len, the slots of the matched path to slots_out (host,
 * capacity n; may be NULL) and the deepest matched node to *last (root when
 * nothing matched).  Stamps the matched path as used now; a node matched
 * only partly is split so that the stamp covers whole nodes.
 * [bhfrc.com §3.1; "SGLang 深度拆解" §2.3 match_prefix; "SGLang 深度解读" §1] */
int sgl_tree_match(sgl_tree* tree, const int32_t* tokens, int64_t n,
                   int64_t* matched_len, int32_t* slots_out, sgl_node* last);

/* Insert the full pages of tokens[0..n) with their slots (host, n entries;
 * the slots of one page must be that page's consecutive slots).  Existing
 * pages are kept; a caller page that differs from the existing page at the
 * same position is a duplicate and is returned to the free list (dup_len
 * counts those tokens).  Nodes are split where the new path diverges.  A
 * trailing partial page is not inserted.  *last = node ending the inserted
 * path (may be NULL).  [bhfrc.com §3.1; "SGLang 深度拆解" §2.3 insert] */
int sgl_tree_insert(sgl_tree* tree, const int32_t* tokens, const int32_t* slots, int64_t n,
                    int64_t* dup_len, sgl_node* last);

/* Add / remove one reference on every node from `node` up to the root.  A
 * referenced node is never evicted.  unlock below zero: SGL_ERR_STATE and
 * nothing changes.  [bhfrc.com §3.2; oripoin.cn "用基数树实现前缀复用"] */
int sgl_tree_lock(sgl_tree* tree, sgl_node node);
int sgl_tree_unlock(sgl_tree* tree, sgl_node node);

/* Slots for n tokens in whole pages popped from the free list, evicting LRU
 * leaves first if the free list is short.  slots_out: host, capacity n
 * (the rest of the last page stays owned by the caller).  SGL_ERR_NO_SLOTS
 * if still short (the evictions that happened stay done). */
int sgl_tree_alloc(sgl_tree* tree, int64_t n, int32_t* slots_out);

/* Return the pages holding slots[0..n) to the back of the free list, each
 * page once, in first-seen order.  For slots a caller owns (not in the tree). */
int sgl_tree_free(sgl_tree* tree, const int32_t* slots, int64_t n);

/* Free at least num_tokens tokens by removing unreferenced leaves, least
 * recently used first (ties: oldest page first), one page at a time from a
 * leaf's end; a parent whose children are gone becomes a leaf.  *freed =
 * tokens freed (less than asked when every remaining leaf is referenced).
 * [oripoin.cn "用基数树实现前缀复用": leaf-first LRU; "SGLang 深度拆解" §2.3 _evict] */
int sgl_tree_evict(sgl_tree* tree, int64_t num_tokens, int64_t* freed);

typedef struct {
    int64_t free_pages;     /* pages on the free list */
    int64_t tree_tokens;    /* tokens held by tree nodes */
    int64_t locked_tokens;  /* tokens of nodes with a reference count > 0 */
    int64_t evictable_tokens; /* tokens of nodes with reference count 0 */
    int64_t num_nodes;      /* tree nodes, root excluded */
    int64_t clock;          /* logical clock (match and insert calls so far) */
} sgl_tree_stats_t;
int sgl_tree_stats(const sgl_tree* tree, sgl_tree_stats_t* out);

/* ======================================================================== */
/* Batch tables: req_to_token + prefix groups                               */
/* ======================================================================== */

typedef struct sgl_groups sgl_groups;

/* View of prefix groups (CSR, library memory).  Segment s covers positions
 * [seg_begin[s], seg_end[s]) of every member request; all members hold the
 * same slots there, so the K/V rows are read from the representative row
 * seg_row[s] (its smallest member).  Members of s are
 * seg_members[seg_member_ptr[s] .. seg_member_ptr[s+1]), ascending.
 * Segments are ordered by (seg_row, seg_begin).  Each position of each
 * request lies in exactly one of its segments.
 * [bhfrc.com §1.3 and §3.1: requests sharing a path are branches of one
 * tree, the shared path computed once] */
typedef struct {
    int32_t num_segments;
    int32_t num_members;
    const int32_t* seg_begin;
    const int32_t* seg_end;
    const int32_t* seg_row;
    const int32_t* seg_member_ptr;
    const int32_t* seg_members;
} sgl_prefix_groups;

/* Build one batch: for each request r in order, match its tokens, lock the
 * match, allocate slots for the unmatched tail, write row r of req_to_token
 * (host [B, ld], ld >= every len; entries past len[r] set to -1), insert the
 * full pages, lock the new last node and release the temporary lock.
 * seq_lens[r] = len[r]; prefix_lens[r] = matched length; last_nodes[r] =
 * the node the request holds a reference on (release it with
 * sgl_tree_finish).  The slots of a trailing partial page (page_size > 1)
 * are private to the request.  If groups_out != NULL, *groups_out receives
 * the batch's prefix groups (create it first with sgl_groups_create; it is
 * refilled).  SGL_ERR_NO_SLOTS: every lock this call took is released and
 * the private pages it allocated are freed; inserted nodes stay as cache.
 * tokens: host array of B host pointers; len: host [B]; the other outputs
 * host [B].  prefix_lens, last_nodes may be NULL.
 * ["SGLang 深度解读" sections "2. Scheduler" and "5. Attention 层"] */
int sgl_build_batch(sgl_tree* tree, int32_t B, const int32_t* const* tokens, const int64_t* len,
                    int32_t* req_to_token, int64_t ld, int32_t* seq_lens, int32_t* prefix_lens,
                    sgl_node* last_nodes, sgl_groups* groups_out);

/* A request is done: unlock its last node and free its private tail page
 * (row: host, its req_to_token row; len: its length). */
int sgl_tree_finish(sgl_tree* tree, sgl_node last, const int32_t* row, int64_t len);
/* sgl_tree_finish for requests 0 .. B-1 in order (a batch from
 * sgl_build_batch): last host [B], req_to_token host [B, ld], seq_lens host
 * [B].  Stops at the first error and returns it (earlier requests stay
 * finished). */
int sgl_tree_finish_batch(sgl_tree* tree, int32_t B, const sgl_node* last, const int32_t* req_to_token, int64_t ld,
                          const int32_t* seq_lens);

/* One decode step of a running batch (after sgl_build_batch): request r
 * gains one token at position seq_lens[r].  Its slot is the first slot of
 * a fresh page when seq_lens[r] is a multiple of the page size, else the
 * slot after req_to_token[r, seq_lens[r] - 1] (the request's private tail
 * page).  The step's fresh pages come from one allocation (evicting LRU
 * leaves if needed) and go to the requests in order.  Writes
 * req_to_token[r, seq_lens[r]] and increments seq_lens[r].  The tree is not
 * touched: the new tokens are cached when the request ends
 * (sgl_tree_cache_finished).  If groups != NULL it must hold this batch's
 * prefix groups (from sgl_build_batch or an earlier append); each request's
 * private trailing segment grows by one position, or a private one-position
 * segment is added where its context ended in a shared segment.
 * req_to_token: host [B, ld], seq_lens: host [B], both updated in place.
 * SGL_ERR_INVALID_ARG (a row already ld long, a tail slot that is not
 * followed by a slot of the same page, groups that do not cover the batch)
 * and SGL_ERR_NO_SLOTS change nothing but the cache that allocation
 * evicted.
 * ["SGLang 深度拆解" (chenxutan.com) §1.3 (the CPU scheduler caches a
 * request's sequence when it finishes); CS349D lecture-16 notes §3.1
 * (continuous batching, the prompt inserted at prefill completion)] */
int sgl_batch_append(sgl_tree* tree, int32_t B, int32_t* req_to_token, int64_t ld, int32_t* seq_lens,
                     sgl_groups* groups);

/* A request ends and its sequence is cached: the full pages of tokens[0,
 * len) go into the tree with the slots of row (host, its req_to_token row),
 * resuming at `last` (the node the request holds, whose path must be this
 * sequence's prefix with these slots); duplicate pages go to the free list;
 * then the request's reference is released and a partial tail page freed.
 * *dup_len (may be NULL) = duplicate tokens freed.  SGL_ERR_STATE: `last`
 * is stale or not referenced; SGL_ERR_INVALID_ARG: the path or the slots
 * disagree (nothing changed). */
int sgl_tree_cache_finished(sgl_tree* tree, sgl_node last, const int32_t* tokens, const int32_t* row, int64_t len,
                            int64_t* dup_len);
/* sgl_tree_cache_finished for requests 0 .. B-1 in order: tokens host array
 * of B host pointers, last host [B], req_to_token host [B, ld], seq_lens
 * host [B].  Stops at the first error and returns it. */
int sgl_tree_cache_finished_batch(sgl_tree* tree, int32_t B, const int32_t* const* tokens, const sgl_node* last,
                                  const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens);

int sgl_groups_create(sgl_groups** out);
void sgl_groups_destroy(sgl_groups* groups);
int sgl_groups_view(const sgl_groups* groups, sgl_prefix_groups* view);

/* Prefix groups of any slot table (host [B, ld] + host seq_lens [B]),
 * computed from the slots alone: positions shared by the same set of
 * requests with identical slot prefixes. */
int sgl_groups_from_table(const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens, int32_t B,
                          sgl_groups* groups_out);

/* ======================================================================== */
/* Attention                                                                */
/* ======================================================================== */

typedef struct {
    int32_t dtype;          /* SGL_DTYPE_F32 or SGL_DTYPE_BF16 (Q, K, V, O), or SGL_DTYPE_BF16_FP8KV */
    int32_t batch;          /* B: requests */
    int32_t num_qo_heads;   /* Hq */
    int32_t num_kv_heads;   /* Hkv */
    int32_t head_dim;       /* d: 64 or 128 */
    int32_t page_size;      /* P >= 1 (addressing is per slot; informative) */
    int64_t num_slots;      /* S: rows of each pool buffer; S * Hkv < 2^31 */
    float sm_scale;         /* <= 0: 1/sqrt(d) */
    int32_t num_sms;        /* planning target; <= 0: query the current device (152 if none) */
    /* extend only: host copies of prefix_lens / extend_lens (B entries)
     * used to size the launch; they must equal the device arrays. */
    const int32_t* host_prefix_lens;
    const int32_t* host_extend_lens;
    /* SGL_DTYPE_BF16_FP8KV only: dequantisation scales of the K and V pools */
    float k_scale;
    float v_scale;
} sgl_attn_params;

typedef struct sgl_plan sgl_plan;

/* Decode planning (host).  Splits every (segment, KV head) into KV chunks
 * and member blocks so that the work items fill the GPU, and lays out the
 * fp32 partial (O, LSE) buffer and the per-request merge lists.  seq_lens:
 * host [B]; groups: the batch's prefix groups.  *workspace_bytes = device
 * workspace the call needs (plan tables + partials + error word).
 * Segments whose end exceeds their representative's seq_len:
 * SGL_ERR_INVALID_ARG.
 * A plan stays valid for later decode calls on the same batch after its
 * requests have grown at their ends (sgl_batch_append): each request's last
 * piece -- over its own trailing positions, or an empty piece at its end
 * when its context ends in a shared segment -- reads up to the request's
 * device seq_len at run time (bounded by ld; a length below the planned
 * one sets error bit 1).  Growth lengthens only those pieces, so the work
 * balance of a reused plan degrades slowly; any other change of the batch
 * (requests added or removed, a different sharing) needs a new plan.
 * [decode steps of a running batch: "SGLang 深度拆解" (chenxutan.com) §1.3;
 * the scheduler prepares the next batch ahead of the GPU: CS349D
 * lecture-16 notes §2.2] */
int sgl_decode_plan(const sgl_attn_params* params, const int32_t* seq_lens, const sgl_prefix_groups* groups,
                    sgl_plan** plan_out, size_t* workspace_bytes);
void sgl_plan_destroy(sgl_plan* plan);

typedef struct {
    int32_t num_items;          /* decode work items (all kinds) */
    int32_t num_wide_items;     /* of which shared-segment tiles (tensor-core tile kernel) */
    int32_t num_partial_rows;   /* fp32 partial (O, LSE) rows */
    int32_t num_merge_entries;  /* partial rows named by the merge lists */
    int32_t chunk_tokens;       /* KV positions per chunk chosen by the planner */
    int64_t upload_bytes;       /* bytes sgl_plan_upload copies host -> device */
    int64_t workspace_bytes;    /* device workspace the plan needs */
} sgl_plan_info_t;
/* Sizes of a plan (host; no device access). */
int sgl_plan_info(const sgl_plan* plan, sgl_plan_info_t* out);

/* Copy the plan's device tables into the head of the workspace
 * (device, >= workspace_bytes, 256-byte aligned) on `stream`, and clear its
 * error word.  Needed once after each sgl_decode_plan before decode calls
 * that use the plan; the plan must stay alive until the copy has run.
 * The attention kernels read these tables before their programmatic
 * dependency wait (while the previous kernel in the stream may still run),
 * so nothing but this call may write the table region of the workspace. */
int sgl_plan_upload(const sgl_plan* plan, void* workspace, size_t ws_bytes, sgl_stream_t stream);

/* Decode attention for B requests, one query token each.
 *   q            device [B, Hq, d] (dtype)
 *   k_pool,v_pool device [num_slots, Hkv, d] (dtype)
 *   req_to_token device int32 [B, ld]
 *   seq_lens     device int32 [B]
 *   plan         from sgl_decode_plan on the same batch, uploaded into workspace
 *                (an MLA plan: SGL_ERR_INVALID_ARG)
 *   o            device [B, Hq, d] (dtype);  lse  device fp32 [B, Hq]
 * Each (segment, KV head) chunk is read from HBM once for all member
 * requests and all query heads of that KV head (GQA packing); the partial
 * (O, LSE) of every chunk are merged per (request, head) by log-sum-exp.
 * A request with seq_len 0 gets O = 0, LSE = -inf. */
int sgl_decode_attn(const void* q, const void* k_pool, const void* v_pool, const int32_t* req_to_token,
                    int64_t ld, const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse,
                    void* workspace, size_t ws_bytes, sgl_stream_t stream);

/* One decode step from host memory, in one call: copy in_bytes from
 * in_host (host memory, pinned for an asynchronous copy) to in_dev (device),
 * run sgl_decode_attn with the given device pointers -- which normally
 * point into in_dev: the step's q, its req_to_token rows and seq_lens staged
 * together -- and copy out_bytes from out_dev (device, normally holding o
 * and lse) to out_host, all queued on `stream` in that order.  in_bytes or
 * out_bytes may be 0 (that copy is skipped).  The caller waits on the stream
 * (or an event recorded after the call) before reading out_host, and must
 * not rewrite in_host before the input copy has run.  Every argument check
 * of sgl_decode_attn, and in_host/in_dev (out_dev/out_host) present when
 * in_bytes (out_bytes) is not 0, is made before any GPU work: on a refusal
 * nothing is queued.
 * [a decode step's metadata prepared on the CPU and moved to the device
 * while the GPU runs the step before: CS349D lecture-16 notes §2.2;
 * "SGLang 深度解读" (luoboask.github.io) section 2, Scheduler] */
int sgl_decode_step(const void* in_host, void* in_dev, size_t in_bytes, const void* q, const void* k_pool,
                    const void* v_pool, const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens,
                    const sgl_plan* plan, void* o, float* lse, const void* out_dev, void* out_host, size_t out_bytes,
                    void* workspace, size_t ws_bytes, sgl_stream_t stream);

/* ---------------------------------------------------------------------
 * MLA grouped decode (CS349D lecture-16 notes, SGLang case study: §4 "More
 * engineering", DeepSeek's MLA with the decompression matrices absorbed
 * into the query and output projections, attention run in the 576-dim
 * latent space by a grouped decode kernel; §5.1: per token ONE stored row
 * of a 512-dim latent plus a 64-dim position part, a single KV "head" read
 * by every query head).
 *
 * For request r and query head h, with c_j the pool row of position j:
 *   s_j = sm_scale * <q[r,h], c_j>  (all latent_dim + rope_dim elements),
 *   O[r,h] = sum_j softmax(s)_j * c_j[0 : latent_dim],  LSE natural log.
 * Shared prefix segments are read once for all member requests and all
 * query heads (64 query rows per work item: members x heads).
 * --------------------------------------------------------------------- */
typedef struct {
    int32_t batch;              /* B requests */
    int32_t num_qo_heads;       /* Hq: 16, 32, 64 or 128 */
    int32_t latent_dim;         /* 512 (the output width) */
    int32_t rope_dim;           /* 64; a pool row holds latent_dim + rope_dim elements */
    int64_t num_slots;          /* pool rows; num_slots <= INT32_MAX */
    int32_t page_size;          /* >= 1 (slots of a page are consecutive) */
    float sm_scale;             /* 0: 1/sqrt(latent_dim + rope_dim) */
    int32_t num_sms;            /* planning target; 0: the current device's SM count */
} sgl_mla_params;

/* MLA decode planning (host).  Splits every prefix-group segment into
 * member blocks of 64 / min(Hq, 64) requests (min(Hq, 64) query heads each)
 * and KV chunks so that the work items fill the GPU, and lays out the fp32
 * partial (O, LSE) rows and the per-(request, head group) merge lists.
 * seq_lens: host [B].  *workspace_bytes as for sgl_decode_plan.  The plan
 * works only with sgl_mla_decode_attn (and sgl_plan_upload / _info /
 * _destroy).  Shapes other than the ones listed: SGL_ERR_UNSUPPORTED;
 * malformed groups: SGL_ERR_INVALID_ARG. */
int sgl_mla_decode_plan(const sgl_mla_params* params, const int32_t* seq_lens, const sgl_prefix_groups* groups,
                        sgl_plan** plan_out, size_t* workspace_bytes);

/* MLA decode attention, one query token per request.
 *   q            device bf16 [B, Hq, latent_dim + rope_dim] (absorbed queries)
 *   kv_pool      device bf16 [num_slots, latent_dim + rope_dim]
 *   req_to_token device int32 [B, ld];  seq_lens device int32 [B]
 *   plan         from sgl_mla_decode_plan on the same batch, uploaded into workspace
 *   o            device bf16 [B, Hq, latent_dim];  lse device fp32 [B, Hq]
 * Slots outside the pool are skipped and flagged in the workspace error
 * word (sgl_check).  A request with seq_len 0 gets O = 0, LSE = -inf.
 * A plan from sgl_decode_plan: SGL_ERR_INVALID_ARG. */
int sgl_mla_decode_attn(const void* q, const void* kv_pool, const int32_t* req_to_token, int64_t ld,
                        const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse, void* workspace,
                        size_t ws_bytes, sgl_stream_t stream);

/* Device workspace needed by sgl_extend_attn for these params (bytes). */
int sgl_extend_workspace_bytes(const sgl_attn_params* params, size_t* bytes);

/* Extend attention (chunked prefill with a cached prefix).
 *   q_new        device [N, Hq, d], N = sum extend_lens; request r's rows
 *                follow request r-1's
 *   prefix_lens, extend_lens  device int32 [B] (equal to the host copies in params)
 *   req_to_token device int32 [B, ld]; the new tokens' K/V are already in
 *                the pool at req_to_token[r, prefix_lens[r] + i]
 *   o            device [N, Hq, d] (dtype);  lse  device fp32 [N, Hq]
 * New token i of request r (position p = prefix_lens[r] + i) attends to
 * positions 0..p of row r.  workspace: device, >= sgl_extend_workspace_bytes,
 * 256-byte aligned; its error word is cleared by this call.
 * ["SGLang 深度解读" "5. Attention 层": K/V written before attention;
 * "SGLang 深度拆解" §3.2 PagedPrefill: skip the cached prefix's compute] */
int sgl_extend_attn(const void* q_new, const void* k_pool, const void* v_pool, const int32_t* req_to_token,
                    int64_t ld, const int32_t* prefix_lens, const int32_t* extend_lens,
                    const sgl_attn_params* params, void* o, float* lse, void* workspace, size_t ws_bytes,
                    sgl_stream_t stream);

/* ---------------------------------------------------------------------------
 * Cache-aware scheduling simulation (host) over the radix tree.
 * A round-based serving loop: every round, requests that have arrived join
 * the waiting queue; the queue is ordered (FCFS: arrival order; LPM: longest
 * cached prefix first, ties in queue order -- the match lengths are taken with
 * sgl_tree_match, which also refreshes the matched nodes' LRU stamps); requests
 * are admitted in that order while fewer than max_running run: the cached
 * prefix is matched and locked, and slots for the rest of the prompt and all
 * of the output are allocated (evicting LRU leaves); an allocation failure
 * ends admission for the round.  Under LPM with defer_tokens > 0 a request is
 * skipped for the round if a request admitted in the same round has the same
 * cached length and the same next min(defer_tokens, uncached) prompt tokens
 * (its prefix will be cached once that one is prefilled).  Then up to
 * prefill_budget prompt tokens are prefilled, in admission order (chunked
 * prefill); a request whose prompt is complete inserts the prompt into the
 * tree now (SGL_INSERT_AT_PREFILL) or only at its end (SGL_INSERT_AT_FINISH).
 * Every request whose prefill completed in an earlier round decodes one
 * output token; after its last token the whole sequence is inserted, its
 * references are released and a partial tail page is freed.  A request with
 * depends_on = j arrives `delay` rounds after request j finishes (a later
 * turn of a conversation).
 * The tree is used and modified as a real scheduler would (its contents
 * afterwards are the cache after the trace).
 * Returns SGL_ERR_STATE if max_rounds pass before every request finished.
 * ["SGLang：从前端 DSL 到 SRT 服务运行时" "用基数树实现前缀复用": cache-aware
 * scheduling by longest shared prefix, leaf-first LRU eviction, reference
 * counts; CS349D lecture-16 notes §3.1-3.3: continuous batching, chunked
 * prefill budget, longest-prefix-first with deferral, insertion at prefill
 * completion] */
enum { SGL_SCHED_FCFS = 0, SGL_SCHED_LPM = 1 };
enum { SGL_INSERT_AT_PREFILL = 0, SGL_INSERT_AT_FINISH = 1 };

typedef struct {
    int32_t policy;          /* SGL_SCHED_FCFS or SGL_SCHED_LPM */
    int32_t insert_at;       /* SGL_INSERT_AT_PREFILL or SGL_INSERT_AT_FINISH */
    int64_t prefill_budget;  /* prompt tokens prefilled per round, >= 1 */
    int32_t max_running;     /* requests running at once, >= 1 */
    int32_t defer_tokens;    /* LPM deferral window, >= 0 (0: off) */
    int64_t max_rounds;      /* guard, >= 1 */
} sgl_sim_config;

typedef struct {
    const int32_t* prompt;   /* host, prompt_len tokens (>= 1) */
    int64_t prompt_len;
    const int32_t* output;   /* host, the output_len tokens it generates (>= 1) */
    int64_t output_len;
    int64_t arrive_round;    /* used when depends_on < 0 (>= 0) */
    int32_t depends_on;      /* -1, or an earlier request index */
    int64_t delay;           /* rounds after depends_on finishes (>= 0) */
} sgl_sim_request;

typedef struct {
    int64_t arrive_round, admit_round, cached_tokens, prefill_done_round, finish_round;
} sgl_sim_result;

typedef struct {
    int64_t rounds;          /* rounds until every request finished */
    int64_t prompt_tokens;   /* prompt tokens of all requests */
    int64_t cached_tokens;   /* of which found in the tree at admission */
    int64_t prefill_tokens;  /* prompt tokens prefilled (= prompt - cached) */
    int64_t decode_tokens;   /* output tokens decoded */
    int64_t evicted_tokens;  /* tree tokens evicted by admissions */
} sgl_sim_stats;

/* reqs, per_req: host arrays of n.  The tree: from sgl_tree_create, with
 * whatever it already caches. */
int sgl_sim_run(sgl_tree* tree, const sgl_sim_config* cfg, int32_t n, const sgl_sim_request* reqs,
                sgl_sim_result* per_req, sgl_sim_stats* stats);

/* Extend attention with the KV write fused in (chunked prefill step).
 *   k_new, v_new device [N, Hkv, d] (dtype), rows ordered like q_new: the
 *                new tokens' K and V, which this call stores into
 *   k_pool, v_pool device [num_slots, Hkv, d] at the slots
 *                req_to_token[r, prefix_lens[r] + i] (caller-owned; the rest
 *                of the pool is only read)
 * Otherwise as sgl_extend_attn, whose result this call equals after the
 * same rows have been written: new token i of request r attends to the
 * cached positions 0..prefix_lens[r]-1 (read from the pool) and to new
 * tokens 0..i (read from k_new / v_new directly in the bf16 path; the fp32
 * and FP8-pool paths write the pool first and read it, so with an FP8 pool
 * the new tokens are seen as their stored E4M3 values).  An out-of-pool slot is not
 * written and sets SGL_ERR_BOUNDS for sgl_check.  Repeated calls over the
 * chunks of a long prompt (prefix_lens = tokens already cached) are a
 * chunked prefill.
 * ["SGLang 深度解读" "5. Attention 层": the new tokens' K/V are stored into
 * token_to_kv_pool at their req_to_token slots before attention;
 * "SGLang：从前端 DSL 到 SRT 服务运行时": chunked prefill] */
int sgl_extend_attn_kvwrite(const void* q_new, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                            const int32_t* req_to_token, int64_t ld, const int32_t* prefix_lens,
                            const int32_t* extend_lens, const sgl_attn_params* params, void* o, float* lse,
                            void* workspace, size_t ws_bytes, sgl_stream_t stream);

/* Wait for `stream`, read the workspace's error word and clear it.
 * SGL_OK, or SGL_ERR_BOUNDS if a kernel skipped an out-of-range slot or a
 * position beyond seq_lens since the word was last cleared. */
int sgl_check(void* workspace, sgl_stream_t stream);

/* Decode attention without a caller-provided workspace.
 * No counterpart on the pages: this is a convenience for callers that cannot
 * allocate device memory -- serving loops whose device memory belongs to
 * another allocator with a fixed budget, or latency-critical paths that avoid
 * cudaMalloc because it can synchronize the device.
 * Same arguments and result as sgl_decode_attn minus the workspace; the
 * plan is uploaded by the call itself.  Scratch is a fixed 64 MiB array in
 * the library's device image, held by every GPU that loads the library
 * until the process exits; a plan whose workspace_bytes exceeds 64 MiB is
 * rejected with SGL_ERR_WORKSPACE, and every other argument error is
 * returned, before any GPU work.  The first call on a device looks the
 * array's address up (cudaGetSymbolAddress, with that device current) and
 * caches it; a device reset (cudaDeviceReset) is not supported afterwards.
 * Each call copies the plan's tables from the plan's host memory, so the
 * call is not meant for stream capture (a captured copy would re-read that
 * memory at every replay): graphs capture sgl_decode_attn with a workspace
 * uploaded beforehand by sgl_plan_upload.  All calls share the
 * array, whose contents are the last call's (each call rewrites the plan
 * tables and clears the error word and merge counters itself): calls that
 * may overlap on the GPU (different streams, or before the previous call
 * has finished reading it) race and must not be issued.  Out-of-range
 * slots are skipped as in sgl_decode_attn, but their error word cannot be
 * read back (there is no workspace pointer to give sgl_check).
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
int sgl_decode_attn_noalloc(const void* q, const void* k_pool, const void* v_pool, const int32_t* req_to_token,
                            int64_t ld, const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse,
                            sgl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SGLATTN_H */
