/*
 * forkkv.h — C ABI of libforkkv: ResidualAttention over a disaggregated,
 * copy-on-write KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation (ForkKV: Scaling Multi-LoRA Agent Serving via Copy-on-Write
 * Disaggregated KV Cache — L2, sections 2, 3, 4 and 7):
 *   a LoRA-adapted key/value projection is xW + xA_i B_i, so the cache is kept
 *   in two parts: a base cache ("bCache": xW_k with RoPE already applied, and
 *   xW_v), shared by every agent that forked from the same prefix, and a rank-r
 *   residual cache ("rCache": xA_k and xA_v, stored without RoPE) private to
 *   each agent.  Attention rebuilds, on chip and never in HBM,
 *       K_j = Kb_j + RoPE_{p_j}(Kr_j B_k[:, hD:(h+1)D])     (deferred RoPE)
 *       V_j = Vb_j + Vr_j B_v[:, hD:(h+1)D]
 *   and returns softmax(q K^T / sqrt(D)) V, evaluating the value path as
 *   sum_j p_j Vb_j + (sum_j p_j Vr_j) B_v so that B_v is applied once per
 *   query after the key loop (associativity of the value path).
 * Fork and copy-on-write follow ForkKV L2 section 3 (Figure 6: a new agent maps
 * the parent's bCache pages and allocates only its own rCache pages) and the
 * ForkServe README ("Design vs APC", "Methods", "Status": fork aliases the
 * parent's page frames with refcounts; the unaligned tail is packed by copying
 * its n_valid rows, not a whole page).
 *
 * Conventions
 *   - Every function returns int32_t: FORKKV_OK (0) or a negative FORKKV_ERR_*.
 *     On error nothing has changed (no allocator state, no launch).
 *   - No C++ exception crosses this boundary.
 *   - Device buffers (pools, page tables, q, out, adapters, tables, workspace)
 *     are allocated and owned by the caller; no entry point allocates device
 *     memory.  The library owns only the host allocator objects it creates.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Kernels run asynchronously: a successful return means the launch was
 *     accepted.  Out-of-range indices met on the device are skipped and
 *     recorded in a device status word read by forkkv_get_device_status().
 *   - Data is bf16 (IEEE binary16 with 8 exponent bits), indices int32.
 *   - Fixed geometry: head_dim D = 128, residual rank r = 16, page size P = 16.
 *
 * Pool layouts (device memory, 16-byte aligned)
 *   Base pools k_base, v_base: [n_layers][num_kv_heads][num_base_pages] tiles of
 *   FORKKV_BASE_TILE_BYTES (head-major, so a run of consecutive page ids of one
 *   head is one contiguous range that a single bulk copy can move).  A tile holds the 16 rows x 128 bf16 of one page and
 *   one KV head in the tensor core's 128-byte-swizzled K-major layout: element
 *   (row t, column d) lives at byte
 *       (d / 64) * 2048 + t * 128 + ((((d % 64) / 8) ^ (t % 8)) * 16) + (d % 8) * 2.
 *   Residual pools k_res, v_res: [n_layers][num_res_pages] tiles of
 *   FORKKV_RES_TILE_BYTES, 16 rows x 16 bf16 in the 32-byte-swizzled layout:
 *       t * 32 + (((k / 8) ^ ((t / 4) % 2)) * 16) + (k % 8) * 2.
 *   A token at logical position j of a sequence lives in row j % 16 of page
 *   table entry j / 16.  forkkv_write_rows() is the portable way to fill pools.
 */
#ifndef FORKKV_H_
#define FORKKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define FORKKV_OK 0
#define FORKKV_ERR_INVALID_ARG (-1)  /* bad size, pointer, alignment or id     */
#define FORKKV_ERR_OUT_OF_PAGES (-2) /* a pool has too few free pages          */
#define FORKKV_ERR_BAD_PAGE (-3)     /* a page id outside its pool             */
#define FORKKV_ERR_REFCOUNT (-4)     /* refcount would underflow               */
#define FORKKV_ERR_UNSUPPORTED (-5)  /* geometry other than D=128, r=16, P=16  */
#define FORKKV_ERR_CUDA (-6)         /* a CUDA runtime call failed             */
#define FORKKV_ERR_SCRATCH (-7)      /* needs more than the static decode scratch */

/* device status bits (forkkv_get_device_status) */
#define FORKKV_DEV_BAD_PAGE 1u  /* a page id read from a device table was out of range */
#define FORKKV_DEV_TIMEOUT 2u   /* a bounded wait on an mbarrier gave up               */
#define FORKKV_DEV_BAD_ARG 4u   /* a device-side argument (length, position) invalid   */

/* ---- fixed geometry ---------------------------------------------------- */
#define FORKKV_PAGE_SIZE 16
#define FORKKV_HEAD_DIM 128
#define FORKKV_RANK 16
#define FORKKV_MAX_GROUP 8             /* query heads per KV head, at most   */
#define FORKKV_BASE_TILE_BYTES 4096    /* 16 rows x 128 bf16                 */
#define FORKKV_RES_TILE_BYTES 512      /* 16 rows x 16 bf16                  */
#define FORKKV_ROPE_ROW_BYTES 256      /* one position of the rotation table */
#define FORKKV_PLAN_ITEM_INTS 16       /* int32 per decode work item         */
#define FORKKV_PLAN_UNIT_INTS 16       /* int32 per decode unit record       */

/* Message for a status code (static string, owned by the library; never
 * NULL, "unknown status" for a code it does not define).  No counterpart in
 * the pages: error reporting of this library. */
const char* forkkv_strerror(int32_t code);
/* Library ABI version (major * 100 + minor).  No counterpart in the pages. */
int32_t forkkv_version(void);

/* ==== host allocator ======================================================
 * Two page pools: base pages (shared, refcounted) and residual pages
 * (private unless FORKKV_FORK_SHARE_RES).  Each pool has a LIFO free stack
 * that initially pops 0, 1, 2, ...; freeing pushes pages, in logical order,
 * whose refcount reaches 0.  Sequence ids count up from 0 and are not reused.
 * An allocator object is not thread-safe: serialise calls on one object.   */
typedef struct forkkv_alloc forkkv_alloc;

#define FORKKV_JOB_BASE 0  /* copy rows of a base page (all layers, all KV heads, K and V) */
#define FORKKV_JOB_RES 1   /* copy rows of a residual page (all layers, k_res and v_res)  */
#define FORKKV_JOB_BASE_ZERO 2 /* zero rows n_valid..15 of base page dst_page (all layers, heads, K and V) */
#define FORKKV_JOB_RES_ZERO 3  /* zero rows n_valid..15 of residual page dst_page (all layers)             */

/* One copy-on-write job: rows [0, n_valid) of page src_page are copied into
 * page dst_page; rows n_valid..15 of dst_page are left untouched.  A zero job
 * (kind *_ZERO, src_page == dst_page) instead sets rows n_valid..15 of
 * dst_page to zero: rows of a frozen tail page that no token has been written
 * to, which the children's slot maps skip (so that a zero probability never
 * meets a never-written value row). */
typedef struct {
  int32_t src_page;
  int32_t dst_page;
  int32_t n_valid;
  int32_t kind; /* FORKKV_JOB_BASE or FORKKV_JOB_RES */
} forkkv_cow_job;

#define FORKKV_FORK_SHARE_RES 1u   /* child aliases the parent's residual pages too */
#define FORKKV_FORK_FREEZE_TAIL 2u /* unaligned prefix: share the tail page read-only, no copy */

typedef struct {
  int32_t n_seqs;
  int32_t base_live, res_live;     /* pages with refcount > 0 */
  int32_t base_free, res_free;     /* pages on the free stacks */
  int32_t base_shared, res_shared; /* pages with refcount > 1 */
  int64_t base_refsum, res_refsum; /* sum of refcounts */
} forkkv_stats;

/* Create an allocator over the two page pools of ForkKV L2 section 2 (Q2: a
 * shared base cache and per-agent residual caches) and section 3 (Figure 6),
 * paged as in the ForkServe README ("Design vs APC": location-addressed page
 * frames, P = 16 tokens a page): num_base_pages base and num_res_pages
 * residual pages (each >= 1) of page_size tokens (page_size must be 16:
 * UNSUPPORTED otherwise; INVALID_ARG for a count < 1 or out == NULL).  *out
 * owns host memory only (page ids, refcounts, per-sequence tables); the device
 * pools it indexes are the caller's.  Release it with forkkv_alloc_destroy. */
int32_t forkkv_alloc_create(int32_t num_base_pages, int32_t num_res_pages, int32_t page_size,
                            forkkv_alloc** out);
/* Free the host memory of an allocator (every sequence with it); NULL is
 * INVALID_ARG.  Device pools are not touched. */
int32_t forkkv_alloc_destroy(forkkv_alloc* alloc);

/* A root sequence (ForkKV L2 section 3, Figure 6: the parent agent whose
 * prefix later agents fork from) of n_tokens >= 0 tokens with ceil(n/16)
 * private base and residual pages (base pages popped in logical order, then
 * residual ones).  OUT_OF_PAGES (nothing taken) when a pool is short. */
int32_t forkkv_seq_create(forkkv_alloc* alloc, int32_t n_tokens, int32_t* seq_out);

/* Fork (ForkKV L2 section 3, Figure 6; ForkServe "Methods", CoW tree):
 * the child's first prefix_len tokens (0 <= prefix_len <= parent length) are
 * the parent's.  Full base pages are aliased (refcount + 1).  If prefix_len
 * is not a multiple of 16, the child gets a new private base page and a job
 * {parent tail page, new page, prefix_len % 16, FORKKV_JOB_BASE} (the pack
 * path of the ForkServe unaligned tail).  Residual pages covering the prefix
 * are newly allocated (the child's adapter gives it its own xA rows, which the
 * caller writes); with FORKKV_FORK_SHARE_RES full residual pages are aliased
 * and a partial one is copied by a FORKKV_JOB_RES job.  Jobs go to
 * jobs[0 .. *n_jobs) (host memory, jobs_cap entries; at most 2 are made). */
int32_t forkkv_fork(forkkv_alloc* alloc, int32_t parent, int32_t prefix_len, uint32_t flags,
                    int32_t* child_out, forkkv_cow_job* jobs, int32_t jobs_cap, int32_t* n_jobs);

/* Freeze-tail fork (FORKKV_FORK_FREEZE_TAIL; ForkServe README, adaptive
 * unaligned tail: pages_freeze = 1 + k ceil(l / P), one read-only tail page
 * shared by the k children instead of a copy in each; "it needs a fork-aware
 * slot map").  With the flag and prefix_len % 16 = t != 0 the child also
 * aliases the parent's partial tail page (refcount + 1, no copy); the child's
 * slots [prefix_len, next multiple of 16) become a hole that its slot map
 * skips, so its own tokens start on a fresh page, and its residual pages are
 * new (or, with FORKKV_FORK_SHARE_RES, the parent's residual tail page is
 * shared the same way).  The parent keeps writing its later tokens into the
 * same page in place (the children read only its first t rows).  Zero jobs
 * (FORKKV_JOB_*_ZERO) clear the rows of that page no token has been written
 * to yet, and the hole rows of the child's own residual page: run a fork's jobs
 * before writing new rows.  A sequence holds at most one hole: a freeze fork
 * whose prefix spans the parent's hole is a pack fork (the child inherits the
 * parent's hole).  Without an unaligned tail the flag changes nothing.
 *
 * Slots: a sequence's keys occupy slots 0, 1, ... (slot s is row s % 16 of its
 * page s / 16); token p is in slot p, or p + hole_len if the sequence has a
 * hole and p >= hole_start.  Page tables and lengths count slots.
 *
 * Grow a sequence by n_tokens >= 0.  A partial last page that is shared
 * (refcount > 1) is first replaced by a private copy (one job per pool, at
 * most 2) unless it is this sequence's frozen tail page past every child's
 * frozen rows (written in place), then pages covering the new slots are added
 * in logical order. */
int32_t forkkv_append(forkkv_alloc* alloc, int32_t seq, int32_t n_tokens, forkkv_cow_job* jobs,
                      int32_t jobs_cap, int32_t* n_jobs);

/* Drop a sequence (ForkServe README, "Design vs APC": the extra pin on owned
 * frames, so that freeing a parent does not drop a trunk its children still
 * map): every page's refcount - 1; pages reaching 0 are pushed back on their
 * free stack in logical order (base pages, then residual pages).  A child's
 * references keep an aliased trunk alive after its parent is freed.  An
 * unknown or already freed sequence is INVALID_ARG; a refcount that would go
 * below 0 is REFCOUNT (nothing changes in either case). */
int32_t forkkv_free(forkkv_alloc* alloc, int32_t seq);

/* Abort a speculative branch (ForkServe README, "Design vs APC" and "Methods":
 * abort costs the residual, not the trunk): exactly forkkv_free, and the
 * number of base and residual pages that went back to the free stacks (the
 * branch's own pages; aliased trunk pages only lose a reference).  Either
 * count pointer may be NULL. */
int32_t forkkv_abort(forkkv_alloc* alloc, int32_t seq, int32_t* n_base_released, int32_t* n_res_released);

/* LCP commit (ForkServe README, "Methods"): bind the observed token prefix of
 * a branch, abort its siblings, split a mid-page boundary.  In this order:
 *  1. each of siblings[0 .. n_siblings) is freed (forkkv_free, in the order
 *     given; distinct, live, and not seq);
 *  2. seq is truncated to lcp_len (0 <= lcp_len <= its length): its pages
 *     from index ceil(lcp_len / 16) on lose a reference, base pages then
 *     residual pages in logical order, pushed when they reach 0;
 *  3. if lcp_len % 16 != 0 and the boundary page (index ceil(lcp_len/16) - 1)
 *     is still shared (refcount > 1), it is replaced by a new private page and
 *     a job {old, new, lcp_len % 16, kind} copies its committed rows: base
 *     first, then residual (at most 2 jobs, host memory, jobs_cap entries).
 * Siblings are aborted before the split so that a page they alone shared with
 * seq is not copied.  All checks (ids, refcounts, free pages after steps 1-2,
 * jobs_cap) come first: on an error nothing changes. */
int32_t forkkv_commit(forkkv_alloc* alloc, int32_t seq, int32_t lcp_len, const int32_t* siblings,
                      int32_t n_siblings, forkkv_cow_job* jobs, int32_t jobs_cap, int32_t* n_jobs);

/* Length of the longest common prefix of two token id sequences (host
 * memory): the number of tokens of a speculative branch that the observed
 * sequence confirms, the lcp_len of forkkv_commit. */
int32_t forkkv_lcp_len(const int32_t* spec, int32_t n_spec, const int32_t* observed, int32_t n_observed,
                       int32_t* out);

/* Length in tokens of a live sequence (INVALID_ARG for an unknown one). */
int32_t forkkv_seq_len(const forkkv_alloc* alloc, int32_t seq, int32_t* len_out);

/* Per-agent page tables (ForkKV L2 section 3, Figure 6: an agent's bCache
 * pages, aliased from its ancestors, and its own rCache pages; the ForkServe
 * README's context tree maps a branch to the parent's frames plus its own):
 * for seqs[0 .. n), row-major [n][stride] base page ids in bpt and residual
 * page ids in rpt (host memory, caller-owned, n * stride int32 each), entries
 * past a sequence's pages set to -1, and seq_lens[i] = its length in slots
 * (tokens + hole length: the seq_lens the attention calls take).  INVALID_ARG
 * for an unknown sequence or one with more than stride pages. */
int32_t forkkv_page_tables(const forkkv_alloc* alloc, const int32_t* seqs, int32_t n, int32_t stride,
                           int32_t* bpt, int32_t* rpt, int32_t* seq_lens);

/* Slot maps of n sequences (ForkServe README, adaptive unaligned tail: the
 * freeze variant "needs a fork-aware slot map"; host memory, caller-owned,
 * 2 n int32): holes[2 i] = first slot of sequence i's hole, holes[2 i + 1] =
 * its length (0, 0 without a hole); the holes array of the attention calls.
 * INVALID_ARG for an unknown sequence. */
int32_t forkkv_slot_maps(const forkkv_alloc* alloc, const int32_t* seqs, int32_t n, int32_t* holes);

/* Refcount of one page (ForkServe README, "Design vs APC": fork aliases frames
 * with refcounts; ForkKV L2 section 3: a bCache page is shared by every agent
 * that maps it).  kind = FORKKV_JOB_BASE or FORKKV_JOB_RES picks the pool;
 * BAD_PAGE for a page id outside it. */
int32_t forkkv_refcount(const forkkv_alloc* alloc, int32_t kind, int32_t page, int32_t* out);
/* Live, free and shared page counts and refcount sums of both pools (the
 * accounting behind ForkKV L2 section 4's memory ratio M_R = 1/N + r/n and the
 * ForkServe README's "Results" page counts).  The struct type holds the name
 * forkkv_stats, so the call is forkkv_stats_get. */
int32_t forkkv_stats_get(const forkkv_alloc* alloc, forkkv_stats* out);

/* ==== pools ================================================================ */
typedef struct {
  void* k_base;            /* [n_layers][num_kv_heads][num_base_pages][4096 B] */
  void* v_base;            /* same shape                                       */
  void* k_res;             /* [n_layers][num_res_pages][512 B]                 */
  void* v_res;             /* same shape                                       */
  int32_t num_base_pages;
  int32_t num_res_pages;
  int32_t num_kv_heads;    /* 1..16 */
  int32_t n_layers;        /* >= 1; layers are stored back to back */
} forkkv_pool_desc;

/* Scatter n_rows new cache rows into layer `layer` of the pools
 * (ForkKV L2 section 7, disaggregation: base activations and residual
 * activations go to separate pools).  Device inputs:
 *   slot_base[n_rows], slot_res[n_rows]: page * 16 + row, or -1 to skip;
 *   k_base_rows, v_base_rows: bf16 [n_rows][num_kv_heads][128] (keys already rotated);
 *   k_res_rows, v_res_rows:   bf16 [n_rows][16] (unrotated).
 * Pass NULL slot_base (or NULL slot_res) to write only the other part. */
int32_t forkkv_write_rows(const forkkv_pool_desc* pools, int32_t layer, int32_t n_rows,
                          const int32_t* slot_base, const int32_t* slot_res,
                          const void* k_base_rows, const void* v_base_rows,
                          const void* k_res_rows, const void* v_res_rows, void* stream);

/* Residual rows of agents forked from a prefix (ForkKV L2 section 3, Figure 6:
 * a child allocates only residual pages and fills them with its own xA rows;
 * section 2 Q2: a LoRA projection is xW + xA B).  For each agent a < n_agents
 * and token t < n_tok:
 *   k_res = x[t] . A[a][0][r]  and  v_res = x[t] . A[a][1][r]  for r < 16,
 * accumulated in fp32 and rounded to bf16 (nearest even), written to the
 * residual slot slot_res[a * n_tok + t] (page = slot / 16, row = slot % 16) of
 * layer `layer`; slot < 0 skips the pair.
 *   x        [n_tok][hidden] bf16, device, 16-byte aligned (the prefix tokens'
 *            inputs of the k and v projections);
 *   A        [n_agents][2][16][hidden] bf16, device, 16-byte aligned (agent a's
 *            LoRA down-projections of the k and v projections, as stored by
 *            PEFT: lora_A.weight is [rank][in_features]);
 *   hidden   a multiple of 8 (>= 8).
 * One launch: the agents are stacked along N of one tensor-core contraction, so
 * x is read once for all of them.  Caller-owned buffers; INVALID_ARG for a bad
 * size, pointer or alignment; a slot past the pool sets FORKKV_DEV_BAD_PAGE. */
int32_t forkkv_residual_fill(const forkkv_pool_desc* pools, int32_t layer, const void* x, int32_t n_tok,
                             int32_t hidden, const void* A, int32_t n_agents, const int32_t* slot_res, void* stream);

/* Decode-step append, fused (one launch): for each new token i < n_rows, its
 * base rows as forkkv_write_rows writes them (slot_base, k_base_rows,
 * v_base_rows; skipped when slot_base is NULL) and its residual rows computed
 * from its hidden state: k_res = x[i] . A[ad][0][r], v_res = x[i] . A[ad][1][r]
 * with ad = adapter_ids[i] (NULL: ad = i), fp32 accumulation, bf16 (nearest
 * even), written at slot_res[i] (skipped when slot_res is NULL).
 *   x [n_rows][hidden], A [n_adapters][2][16][hidden] bf16, device, 16-byte
 *   aligned, hidden a multiple of 8; an adapter id outside [0, n_adapters)
 *   sets FORKKV_DEV_BAD_ARG and uses adapter 0. */
int32_t forkkv_append_rows(const forkkv_pool_desc* pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                           const int32_t* slot_res, const void* k_base_rows, const void* v_base_rows, const void* x,
                           int32_t hidden, const void* A, int32_t n_adapters, const int32_t* adapter_ids,
                           void* stream);

/* Execute copy-on-write jobs on every layer (ForkServe "Status": the pack path
 * copies n_valid rows of a page, not the page).  `jobs` is HOST memory; the
 * jobs travel in the kernel's parameters, so no device buffer is needed.
 * Base jobs copy K and V of every KV head; residual jobs copy k_res and v_res.
 * Rows >= n_valid of the destination are not written.  Ids and n_valid are
 * checked on the host (BAD_PAGE / INVALID_ARG) before anything is launched. */
int32_t forkkv_cow_copy_rows(const forkkv_pool_desc* pools, const forkkv_cow_job* jobs, int32_t n_jobs,
                             void* stream);

/* ==== rotation table ======================================================
 * cos/sin of p * theta^(-2i/128) for positions p < n_positions and the 64
 * rotate-half frequencies i (bf16), FORKKV_ROPE_ROW_BYTES per position, laid
 * out page-major: frequencies (2m, 2m+1) form the 8-byte group m =
 * [cos 2m, cos 2m+1, sin 2m, sin 2m+1] of position p, at byte
 * (p / 16) * 4096 + (m / 4) * 512 + (p % 16) * 32 + (m % 4) * 8, so that the
 * same groups of consecutive positions are contiguous.
 * Angles are reduced exactly in 64-bit fixed point before sin/cos. */
/* Bytes of a table for n_positions >= 0 positions, whole pages of 16
 * positions (INVALID_ARG for n_positions < 0). */
int32_t forkkv_rope_table_bytes(int32_t n_positions, size_t* bytes);
/* Fill a caller-owned device table (16-byte aligned, forkkv_rope_table_bytes
 * long) with the rotations of ForkKV L2 section 7's deferred RoPE (Algorithm 1
 * line 8, RoPE(K_res B_k) at each key's position), for theta > 0.  One launch
 * on `stream`. */
int32_t forkkv_rope_table_build(double rope_theta, int32_t n_positions, void* table, void* stream);

/* ==== decode work plan =====================================================
 * Splits the key ranges of a decode batch into work items so that pages
 * shared by several agents (a fork tree's trunks) are read once per group of
 * up to 4 agents, and deals the (item, KV head) units over persistent CTAs so
 * that their estimated costs balance.  Built on the host from host copies of
 * the page tables.  Layout, all int32:
 *   items      n_items records of FORKKV_PLAN_ITEM_INTS:
 *              [0] first logical page  [1] end logical page  [2] n_agents (1, 2
 *              or 4)  [3] pages per stage (8)  [4..11] agent indices (slots past
 *              n_agents repeat the first)  [12] first partial slot
 *   slot CSR   n_agents + 1 offsets, then n_slots slots (each agent's partials)
 *   units      n_units = n_items * num_kv_heads records of FORKKV_PLAN_UNIT_INTS,
 *              one per (item, KV head): [0] first logical page  [1] end logical
 *              page  [2] n_agents  [3] KV head  [4] first partial slot  [5] record
 *              of the same CTA's next unit, or -1  [6..9] agent indices  [10..15]
 *              zero.  CTA c of the decode kernel starts at record c (c < n_ctas)
 *              and follows the links. */
typedef struct {
  int32_t n_items;     /* work items */
  int32_t n_slots;     /* partial-result slots */
  int32_t n_ctas;      /* CTAs of the decode kernel (grid size) */
  int32_t n_units;     /* n_items * num_kv_heads */
  int32_t plan_ints;   /* int32 words written to plan */
} forkkv_plan_info;

/* Build a plan (ForkKV L2 section 3, Figure 6 and the ForkServe README's
 * context tree: the trunk of a fork tree is read once for the agents that map
 * it).  bpt_host [n_agents][pt_stride] and seq_lens_host [n_agents] are host
 * copies of the attention call's tables; plan is caller-owned host memory of
 * plan_cap_ints int32 (INVALID_ARG, with info->plan_ints = the size needed,
 * when it is too small).  target_ctas: CTAs to spread the units over (0 = one
 * per SM of the current device); the plan uses at most that many.  Copy the
 * plan to the device and pass it with info's counts in forkkv_attn_params. */
int32_t forkkv_plan_build(const int32_t* bpt_host, const int32_t* seq_lens_host, int32_t n_agents,
                          int32_t pt_stride, int32_t num_kv_heads, int32_t target_ctas,
                          int32_t* plan, int32_t plan_cap_ints, forkkv_plan_info* info);

/* ==== attention ============================================================ */
typedef struct {
  int32_t n_agents;        /* A >= 1 */
  int32_t q_len;           /* 1 for decode; chunk length C for prefill */
  int32_t num_q_heads;     /* Hq = G * num_kv_heads with 1 <= G <= 8 */
  int32_t num_kv_heads;    /* must equal pools.num_kv_heads */
  int32_t head_dim;        /* must be 128 */
  int32_t rank;            /* must be 16  */
  int32_t page_size;       /* must be 16  */
  int32_t layer;           /* layer of the pools to read */
  forkkv_pool_desc pools;
  const void* q;           /* bf16 [A][q_len][Hq][128], already rotated at `positions` */
  void* out;               /* bf16 [A][q_len][Hq][128] */
  const int32_t* bpt;      /* [A][pt_stride] base page ids (device) */
  const int32_t* rpt;      /* [A][pt_stride] residual page ids (device) */
  int32_t pt_stride;
  const int32_t* seq_lens; /* [A] key slots of each agent (forkkv_page_tables), including the query
                              tokens' own rows */
  const int32_t* positions;/* [A][q_len] absolute query positions; the key in slot s is visible iff
                              s < seq_len, s is not in the agent's hole and its position (s, or
                              s - hole_len past the hole) <= the query position */
  int32_t max_seq_len;     /* host-known bound on every seq_len */
  const void* B_k;         /* bf16 [n_adapters][16][num_kv_heads * 128] */
  const void* B_v;         /* bf16 [n_adapters][16][num_kv_heads * 128] */
  const int32_t* adapter_ids; /* [A] adapter of each agent, or NULL for agent a -> adapter a */
  int32_t n_adapters;
  const void* rope_table;  /* table for >= max_seq_len positions (whole pages of 16 are read),
                              or NULL: built in workspace */
  int32_t rope_table_positions;
  double rope_theta;       /* used when rope_table is NULL */
  float sm_scale;          /* 0 -> 1/sqrt(128) */
  const int32_t* plan;     /* device copy of a forkkv_plan_build plan, or NULL (decode only) */
  int32_t plan_items;      /* the plan's n_items, n_slots and n_ctas */
  int32_t plan_slots;
  int32_t plan_ctas;
  void* workspace;         /* device scratch, >= the *_workspace_size bytes, 256-byte aligned */
  size_t workspace_bytes;
  const int32_t* holes;    /* [A][2] device: each agent's slot map (first hole slot, hole length;
                              forkkv_slot_maps), or NULL when no agent has a hole */
} forkkv_attn_params;

/* Scratch bytes forkkv_residual_attn_decode needs for these params (the
 * split-KV partials of ForkKV L2 section 4's attention fusion, one (m, l, acc,
 * acc_r) per work segment, plus the rotation table when p->rope_table is NULL).
 * Validates p as the decode call does (same status codes); *bytes is a
 * multiple of 256. */
int32_t forkkv_decode_workspace_size(const forkkv_attn_params* p, size_t* bytes);

/* ResidualAttention decode (ForkKV L2 section 7, the decode version of the
 * kernel; section 4: deferred RoPE of K_res B_k at each key's position, the
 * attention fusion sum p Vb + (sum p Vr) B_v, and check 6, acc and acc_r
 * rescaled together): q_len = 1, one query token per agent at positions[a]
 * (= seq_lens[a] - 1 for a decode step whose row is already written).
 * Split-KV over pages (or over a plan's items), dual-accumulator online
 * softmax, then one merge per (agent, query head) that applies B_v once and
 * writes bf16 out [A][Hq][128].  Every pointer is the caller's device memory
 * (see forkkv_attn_params); workspace >= forkkv_decode_workspace_size bytes.
 * Host checks (INVALID_ARG / UNSUPPORTED, nothing launched): geometry, null
 * pointers, alignment, workspace size, plan sizes.  Device checks (status
 * word): page ids, lengths, positions, adapter ids.  Asynchronous on `stream`;
 * launches 2 kernels (3 if the rotation table is built in the workspace). */
int32_t forkkv_residual_attn_decode(const forkkv_attn_params* p, void* stream);

/* Scratch bytes the prefill chunk needs (the rotation table when
 * p->rope_table is NULL, else 0); validates p as the prefill call does. */
int32_t forkkv_prefill_workspace_size(const forkkv_attn_params* p, size_t* bytes);

/* ResidualAttention over a prefill chunk (ForkKV L2 section 7, the prefill
 * version of the kernel; the same deferred RoPE and fusion as decode): q_len
 * query tokens per agent at `positions` [A][q_len], causal (key j visible iff
 * its position <= the query position and j < seq_len), out [A][q_len][Hq][128].
 * The chunk's own rows must already be in the pools (forkkv_write_rows).  A
 * query position outside [0, seq_len) sets FORKKV_DEV_BAD_ARG.  Same
 * ownership, host checks and device checks as the decode call. */
int32_t forkkv_residual_attn_prefill_chunk(const forkkv_attn_params* p, void* stream);

/* ==== decode without caller scratch =======================================
 * No counterpart in the paper: an addition for callers that cannot allocate.
 * Some callers own no spare device memory to lend as scratch (a serving engine
 * that gives nearly all free HBM to its own KV-cache pool at start-up, or a
 * plugin host that calls an attention op without offering a workspace and
 * forbids cudaMalloc on its hot path, since an allocation can synchronise the
 * device and can fail under memory pressure).  This entry point computes
 * exactly what forkkv_residual_attn_decode computes, with the same arguments,
 * but keeps its scratch in a fixed array of FORKKV_STATIC_SCRATCH_BYTES inside
 * the library's device image, which every GPU that loads the library holds
 * until the process exits.  The workspace fields of `p` are ignored; nothing
 * is allocated (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - Workloads whose scratch (forkkv_decode_workspace_size, which includes the
 *     rotation table when `p->rope_table` is NULL) exceeds the array are
 *     rejected with FORKKV_ERR_SCRATCH before anything is launched.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and caches it per device ordinal; make that first
 *     call before any stream capture.  The cached address belongs to the
 *     device's primary context: after cudaDeviceReset the process must not
 *     call this entry point again (the same holds for the status word that
 *     forkkv_get_device_status reads).
 *   - Every call shares the one array and leaves its contents behind; nothing
 *     in it needs to start at zero (every partial is written before it is read).
 *     Calls whose kernels overlap on the GPU (different streams without
 *     ordering, or concurrent host threads) race on the array: serialise them. */
#define FORKKV_STATIC_SCRATCH_BYTES (8u << 20)
int32_t forkkv_residual_attn_decode_static(const forkkv_attn_params* p, void* stream);

/* ==== one model decode step as one CUDA graph ==============================
 * ForkKV L2 section 5 reports decode throughput per model step (decode batch
 * across all layers); one step of an n_layers model is, per layer l in order,
 * the write of that step's new rows (forkkv_write_rows with rows[l], skipped
 * when rows is NULL or rows[l].n_rows == 0) and forkkv_residual_attn_decode
 * (params[l]).  forkkv_step_graph_create captures that sequence once, on a
 * private stream, into a CUDA graph; forkkv_step_graph_launch replays it on
 * `stream` with one launch call.
 *   - Everything is validated as the per-layer calls validate it; any error
 *     ends the capture and returns that status with *out unchanged.
 *   - The graph records addresses, sizes and the decode geometry (n_agents,
 *     max_seq_len, the plan and its CTA count): between launches the caller
 *     may change the contents of every buffer (q, new rows, slots, page
 *     tables, seq_lens, positions) but not where they are nor the geometry;
 *     a step that needs a longer max_seq_len or a new plan (a sequence that
 *     enters a new page) needs a new graph.
 *   - The graph owns only its CUDA graph objects; every buffer stays the
 *     caller's and must outlive it.  Release it with forkkv_step_graph_destroy.
 *   - Make one ordinary call of forkkv_write_rows and forkkv_residual_attn_decode
 *     on the device first (it resolves kernel attributes and the status word). */
typedef struct {
  int32_t n_rows;            /* new rows of this layer (one per agent in a decode step) */
  const int32_t* slot_base;  /* [n_rows] device, or NULL (no base rows) */
  const int32_t* slot_res;   /* [n_rows] device, or NULL (no residual rows) */
  const void* k_base_rows;   /* [n_rows][Hkv][128] bf16 device */
  const void* v_base_rows;
  const void* k_res_rows;    /* [n_rows][16] bf16 device */
  const void* v_res_rows;
} forkkv_step_rows;

typedef struct forkkv_step_graph forkkv_step_graph;

int32_t forkkv_step_graph_create(const forkkv_attn_params* params, const forkkv_step_rows* rows, int32_t n_layers,
                                 forkkv_step_graph** out);
int32_t forkkv_step_graph_launch(forkkv_step_graph* graph, void* stream);
int32_t forkkv_step_graph_destroy(forkkv_step_graph* graph);

/* Self-test of the bounded device waits.  The pages have no counterpart: this
 * serves the failure handling of the library itself.  Every wait inside the
 * kernels (on an mbarrier that a copy, a tensor-core commit or another warp
 * completes) polls a bounded number of times; if the event never comes it gives
 * up, sets FORKKV_DEV_TIMEOUT in the device status word and the kernel winds
 * down instead of hanging the GPU.  This call launches one tiny kernel whose
 * thread waits, through the same wait routine, on an mbarrier that nothing ever
 * completes, giving up after `polls` polls (1 .. 1048576; each poll may suspend
 * the thread for a hardware-chosen time of the order of a microsecond).  The
 * kernel returns normally, so the context stays usable; a following
 * forkkv_get_device_status() reports FORKKV_DEV_TIMEOUT.  `polls` out of range:
 * FORKKV_ERR_INVALID_ARG, nothing launched.  Allocates nothing. */
int32_t forkkv_wait_selftest(uint32_t polls, void* stream);

/* Read and clear the device status word of the current device (OR of
 * FORKKV_DEV_* bits set by kernels since the last read).  Synchronises
 * `stream`.  No counterpart in the pages: the library's failure reporting
 * (bad page ids, lengths or positions met on the device, and bounded waits
 * that gave up, are recorded here instead of faulting or hanging). */
int32_t forkkv_get_device_status(uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FORKKV_H_ */
