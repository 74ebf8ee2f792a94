/*
 * dsakv.h -- C ABI of the decode-step KV path of DeepSeek-Sparse-Attention
 * style serving with host-offloaded KV and a set-associative FIFO device pool,
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources the operations follow:
 *   [GLM] "GLM-5.2 shared-Indexer KV Cache Offload" (CANN cann-recipes-infer
 *         guide): §2.1 Lightning-Indexer top-k and sparse flash attention,
 *         §4.2 shared planning, §4.3 set-associative FIFO pool, §4.4 SFA first
 *         and refill later, §5 the DsaPlan / DsaServe / DsaInstall split,
 *         §5.1 model-side orchestration.
 *   [TS]  "TokenSpeed" engine audit, MLA kernel section: the latent row
 *         (512 latent + 64 rope values) is stored once and serves as K and V.
 *
 * Shapes: B requests, k selected positions per request, S sets of W ways
 * (pool of P = S*W entries per request and layer), H query heads, latent
 * rows of D = 576 bf16 values (1152 bytes: 512 latent + 64 rope).
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every buffer. The library keeps no state
 *     between calls and allocates no memory (workspaces are passed in).
 *   - Pointers are device pointers unless stated otherwise; host KV is pinned
 *     host memory, passed as the device-accessible address of that memory
 *     (see ts_host_register).
 *   - Streams: a call only enqueues work on `stream`; it never synchronizes.
 *     Ordering between streams is the caller's (events).
 *   - Errors: shapes, sizes and alignment are checked on the host before
 *     anything is launched (TS_ERR_INVALID_ARG / TS_ERR_UNSUPPORTED /
 *     TS_ERR_WORKSPACE, nothing enqueued). A failed launch returns
 *     TS_ERR_CUDA. Data found wrong on the device (an id outside the context,
 *     a slot outside the pool, a NaN score, a wait that gave up) sets bits of
 *     the caller's int32 error word `err` (TS_DEVERR_*) and the offending
 *     element is skipped; nothing traps. `err` may be NULL to skip reporting.
 *     The caller clears it and reads it after the stream's work completes
 *     (ts_read_error does both the wait and the read).
 */
#ifndef DSAKV_H
#define DSAKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = -1,
  TS_ERR_UNSUPPORTED = -2,
  TS_ERR_WORKSPACE = -3,
  TS_ERR_CUDA = -4,
  TS_ERR_DEVICE_CHECK = -5
} ts_status;

/* Bits of the device error word. */
#define TS_DEVERR_ID_RANGE 0x01   /* token id outside [0, ctx_len) */
#define TS_DEVERR_NAN 0x02        /* NaN indexer score */
#define TS_DEVERR_SLOT_RANGE 0x04 /* pool slot / selection position out of range */
#define TS_DEVERR_PTR_RANGE 0x08  /* FIFO pointer outside [0, W) */
#define TS_DEVERR_CTX 0x10        /* ctx_len outside [k, max_ctx] */
#define TS_DEVERR_TIMEOUT 0x20    /* a bounded wait inside a kernel gave up */
#define TS_DEVERR_COUNT 0x40      /* a selection did not come out at size k */
#define TS_DEVERR_ORDER 0x80      /* ids not strictly ascending where a call needs them so */

#define TS_D 576        /* values per latent row */
#define TS_D_LATENT 512 /* latent ("nope") part, also the V part */

/* Text for a status code (static storage). */
const char* ts_status_string(ts_status status);

/* Page-lock and map caller-owned host memory [host, host + bytes) so that
 * kernels can read it in place (zero-copy), and return the device-accessible
 * address in *dev. Pair with ts_host_unregister. Host only; no device work. */
ts_status ts_host_register(void* host, size_t bytes, void** dev);
ts_status ts_host_unregister(void* host);

/* Allocate `bytes` of page-locked host memory mapped for the device
 * (cudaHostAlloc), returning its host address in *host and its
 * device-accessible address in *dev; pair with ts_host_free. Measured on
 * GB300: zero-copy gathers read such memory 5-10 % faster than registered
 * memory, and more evenly. Do not use it as the source of DMA copies while
 * gathers run: after a large DMA from it, zero-copy reads stalled for a while
 * (use registered memory and ts_copy for that). Host only. */
ts_status ts_host_alloc(size_t bytes, void** host, void** dev);
ts_status ts_host_free(void* host);

/* Copy `bytes` bytes from src to dst with the SMs (16-byte loads and stores).
 * Either side may be device memory or registered host memory (its device-
 * accessible address). For moving a step's inputs and outputs across the host
 * link: on GB300 systems, DMA copies from many distinct host buffers were seen
 * to slow the zero-copy gathers that run at the same time, where SM copies
 * were not. Both pointers 16-byte aligned, bytes a multiple of 16. Enqueues
 * on `stream`; no allocation. */
ts_status ts_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* Wait for `stream`, read the error word into *bits (host), clear it on the
 * device. Returns TS_ERR_DEVICE_CHECK when any bit was set. */
ts_status ts_read_error(int32_t* err, int32_t* bits, cudaStream_t stream);

/* Limit, in nanoseconds of the GPU's global timer, of each bounded wait inside
 * the attention kernels launched after this call (their own limit is 2 s);
 * 0 restores it. Process-wide, the library's one setting. For tests of the
 * error path: with a limit shorter than a tile load the attention gives up
 * (TS_DEVERR_TIMEOUT; its output is then undefined), lets every copy it issued
 * land, frees its tensor memory and returns, and the next call with the
 * default limit computes normally. Host only. */
void ts_set_wait_limit_ns(uint64_t ns);

/* ---------------------------------------------------------------------------
 * ts_topk -- top-k of the Lightning-Indexer scores ([GLM] §2.1: the indexer
 * picks the history positions most relevant to the current query; SFA runs on
 * those only).
 *
 *   scores   float  [B][ctx_stride]  row b valid on [0, ctx_len[b])
 *   ctx_len  int32  [B]              device; k <= ctx_len[b] <= max_ctx
 *   ids      int32  [B][k]           out: the k positions of largest score,
 *                                    ties to the lower position, -0.0 == +0.0,
 *                                    in ascending position order
 *   ws       workspace of ts_topk_workspace_size(B, max_ctx, k) bytes,
 *            256-byte aligned, contents need not be preserved
 * Requires scores 16-byte aligned and ctx_stride a multiple of 4, max_ctx <=
 * ctx_stride, 1 <= k <= 8192. A NaN score sets TS_DEVERR_NAN (the NaN ranks
 * lowest); a ctx_len outside [k, max_ctx] sets TS_DEVERR_CTX and that
 * request's ids are all -1.
 * ------------------------------------------------------------------------- */
size_t ts_topk_workspace_size(int B, int max_ctx, int k);
ts_status ts_topk(const float* scores, int64_t ctx_stride, const int32_t* ctx_len,
                  int B, int max_ctx, int k, int32_t* ids, void* ws, size_t ws_bytes,
                  int32_t* err, cudaStream_t stream);

/* ts_topk_noalloc -- ts_topk for callers that cannot allocate device memory
 * (a plugin inside a host engine that owns every allocation, a process whose
 * device memory is reserved before it starts, code that runs where
 * cudaMalloc is not allowed). The pages have no counterpart; it is an
 * interface variant only. Same arguments, results and errors as ts_topk,
 * minus the workspace: the scratch is one fixed device array inside this
 * library (about 34.5 MiB, held on every GPU that loads the library until the
 * process exits). Limits: B <= 128 and B * max_ctx <= 4,194,304; beyond them
 * the call returns TS_ERR_UNSUPPORTED before enqueuing anything. The call
 * allocates nothing. Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture. Every call uses the same array and clears
 * the parts that must start at zero; calls whose work overlaps on the GPU
 * (other streams, other host threads) race on it, so serialize them. */
ts_status ts_topk_noalloc(const float* scores, int64_t ctx_stride, const int32_t* ctx_len,
                          int B, int max_ctx, int k, int32_t* ids, int32_t* err,
                          cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_plan -- the shared plan of an IndexShare group ([GLM] §4.2, §5 DsaPlan;
 * pool policy §4.3). Once per group: classify every selected id as a pool hit
 * or a host miss, list the distinct misses compactly, and choose the slot each
 * miss replaces under the set-associative FIFO policy.
 *
 *   ids        int32 [B][k]   selected token ids (any order, repeats allowed)
 *   ctx_len    int32 [B]      an id t is valid when 0 <= t < ctx_len[b]
 *   pool_tags  int32 [B][P]   token held by each slot, -1 = empty; slot
 *                             s*W + w is way w of set s; token t lives in set
 *                             t mod S
 *   fifo_ptr   int32 [B][S]   per-set FIFO pointer, in [0, W)
 * Outputs (entries at and past miss_count[b] are left untouched):
 *   src_map    int32 [B][k]   hit: the slot (>= 0); miss of token t: -1 - t;
 *                             invalid id: INT32_MIN (and TS_DEVERR_ID_RANGE)
 *   miss_ids   int32 [B][k]   distinct missed tokens, ascending
 *   miss_pos   int32 [B][k]   first position of each missed token in ids
 *   victim     int32 [B][k]   slot the miss replaces: set*W + (ptr + rank) mod W,
 *                             rank = order of the miss among its set's misses
 *   install    uint8 [B][k]   non-zero when the miss survives the step (the
 *                             last W misses of a set); 0 when a later miss of
 *                             the same set in the same step replaces it.
 *                             1: no position of this step reads the victim
 *                             slot (the row may go in as soon as it arrives);
 *                             2: the slot is read as a hit in this step (the
 *                             row goes in only after the layer's reads)
 *   miss_count int32 [B]      distinct missed tokens
 *   miss_rows  int32 [B]      positions that miss (a repeated missed token counts
 *                             at every position; equals miss_count when no
 *                             token repeats)
 *   ptr_next   int32 [B][S]   (ptr + misses in the set) mod W
 * Hits never move a pointer; a hit slot may be chosen as a victim (plain FIFO),
 * which is safe because every layer reads its rows before its own refill.
 * Requires 1 <= W <= 32, P*4 + 12*S + 16*k bytes <= 200 KiB, k <= 4096.
 * ------------------------------------------------------------------------- */
ts_status dsa_plan(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                   const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                   int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                   int32_t* victim, uint8_t* install, int32_t* miss_count,
                   int32_t* miss_rows, int32_t* ptr_next, int32_t* err, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_plan_reuse -- the base design's adjacent-step reuse ([GLM] §2.1
 * GatherSelectionKvCache, §2.2), in the plan's form so that dsa_gather_kv
 * serves it: the device keeps only the previous step's selection buffer
 * (its row i holds the row of prev_ids[i]); a token the previous step also
 * selected is a hit on that row, any other token a miss read from host.
 *
 *   ids       int32 [B][k]   strictly ascending per request (ts_topk's output)
 *   prev_ids  int32 [B][k]   the previous step's ids, strictly ascending;
 *                            -1 marks an empty entry (before the first step)
 *   ctx_len   int32 [B]
 * Outputs as dsa_plan's: src_map (hit: the row in the previous selection,
 * miss of t: -1 - t, invalid: INT32_MIN), miss_ids / miss_pos (ascending),
 * miss_count, miss_rows (= miss_count). Gather with dsa_gather_kv, the
 * previous selection buffer as the pool (P = k). An id outside the context
 * sets TS_DEVERR_ID_RANGE; ids not in strictly ascending order set
 * TS_DEVERR_ORDER (the request's plan is then undefined). k <= 16384.
 * ------------------------------------------------------------------------- */
ts_status dsa_plan_reuse(const int32_t* ids, const int32_t* prev_ids, const int32_t* ctx_len,
                         int B, int k, int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                         int32_t* miss_count, int32_t* miss_rows, int32_t* err,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_plan_lru -- dsa_plan for a fully associative pool of P entries managed
 * least recently used first ([GLM] §3: the 8192-entry device pool the pages
 * measured before adopting the set-associative FIFO of §4.3). A token may sit
 * in any slot. Per step: every selected token already resident is a hit (its
 * slot); the hits are touched in position order, then the distinct misses are
 * installed in ascending id, each into the least recently used slot (empty
 * slots first, lowest index first).
 *
 *   ids        int32 [B][k]   strictly ascending per request (ts_topk's output)
 *   pool_tags  int32 [B][P]   token held by each slot, -1 = empty (in/out)
 *   lru_order  int32 [B][P]   the slots from least to most recently used (in/out;
 *                             a permutation of 0..P-1; a cold pool has every
 *                             tag -1 and the identity order)
 * Outputs as dsa_plan's; every install has code 1 (with k <= P a victim is
 * never a slot the step reads, so the gather may write it on arrival) and no
 * refill is needed. Unlike dsa_plan, the pool's tags and order are updated
 * here, at plan time: nothing else reads them, and the next plan runs after
 * this one. Requires k <= P, k <= 4096, 5 * P + P / 8 + 12 * k bytes <= 200 KiB
 * (P <= 32768 at k = 2048). Ids not strictly ascending set TS_DEVERR_ORDER; an
 * order that is not a permutation of the slots, or a token held by two slots,
 * sets TS_DEVERR_SLOT_RANGE, writes no install and leaves the order as it was
 * (in either case the plan is undefined).
 * ------------------------------------------------------------------------- */
ts_status dsa_plan_lru(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                       int32_t* pool_tags, int32_t* lru_order, int P, int32_t* src_map,
                       int32_t* miss_ids, int32_t* miss_pos, int32_t* victim, uint8_t* install,
                       int32_t* miss_count, int32_t* miss_rows, int32_t* err,
                       cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_gather_kv -- serve one layer's selected rows ([GLM] §5 DsaServe, §5.1;
 * base design §2.1 GatherSelectionKvCache). Row j of request b is copied from
 * the device pool when src_map >= 0 and read in place from pinned host memory
 * (zero-copy) when src_map = -1 - t. The host rows are read first, from the
 * plan's compact miss list (miss_ids / miss_pos / miss_count of dsa_plan for
 * the same ids), so the host-link transfers start at once; the pool rows and
 * any repeated miss follow.
 *
 *   src_map, miss_ids, miss_pos, miss_count, miss_rows   outputs of dsa_plan
 *   pool_l  bf16 [B][P][576]          device, this layer's pool
 *   host_l  bf16 [B][ctx_stride][576] device-accessible address of pinned host
 *                                     memory, this layer's full latent KV
 *   sel_l   bf16 [B][k][576]          out: the selection buffer SFA reads
 * All three 16-byte aligned. Out-of-range slots or host rows set
 * TS_DEVERR_SLOT_RANGE / TS_DEVERR_ID_RANGE and leave that row untouched.
 * ------------------------------------------------------------------------- */
ts_status dsa_gather_kv(const int32_t* src_map, const int32_t* miss_ids,
                        const int32_t* miss_pos, const int32_t* miss_count,
                        const int32_t* miss_rows, int B, int k,
                        const void* pool_l, int P, const void* host_l, int64_t ctx_stride,
                        const int32_t* ctx_len, void* sel_l, int32_t* err,
                        cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_stage_misses -- serve one layer's missed rows into a staged-layout pool
 * ([GLM] §5 DsaServe, §5.1; the hit half of the serve needs no copy here, see
 * sfa_mla_decode_pool). Only the host-link part of the gather: each distinct
 * missed token t of request b, first at position j (dsa_plan's miss_ids /
 * miss_pos / miss_count), is read in place from pinned host memory into
 *   pool_l[b][P + j]
 * and, with victim / install given (both or neither), an install with code 1
 * (no position of the step reads its victim slot) also goes straight into
 *   pool_l[b][victim]
 * as it arrives, leaving the refill only the code-2 installs.
 *
 *   pool_l  bf16 [B][P + k][576]       device, the staged layout: rows 0..P-1
 *                                      of a request are its pool slots, rows
 *                                      P..P+k-1 stage the step's misses
 *   host_l  bf16 [B][ctx_stride][576]  device-accessible address of pinned
 *                                      host memory, this layer's latent KV
 * Both 16-byte aligned; B * (P + k) < 2^31. A bad id or victim sets
 * TS_DEVERR_ID_RANGE / TS_DEVERR_SLOT_RANGE and skips that row.
 * ------------------------------------------------------------------------- */
ts_status dsa_stage_misses(const int32_t* miss_ids, const int32_t* miss_pos,
                           const int32_t* miss_count, const int32_t* victim,
                           const uint8_t* install, int B, int k, void* pool_l, int P,
                           const void* host_l, int64_t ctx_stride, const int32_t* ctx_len,
                           int32_t* err, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_refill_pool -- the deferred refill of one layer's pool ([GLM] §4.4, §5
 * DsaInstall, §5.1). For every installed miss i of request b (install != 0):
 *   pool_l[b][victim[i]] = sel_l[b][miss_pos[i]]   (the missed row's bytes)
 * and, when update_metadata != 0 (the group's last layer):
 *   pool_tags[b][victim[i]] = miss_ids[i];  fifo_ptr[b][:] = ptr_next[b][:].
 * Must run after this layer's dsa_gather_kv (it evicts slots the gather reads)
 * and, with update_metadata, after the refills of every layer of the group.
 * ------------------------------------------------------------------------- */
ts_status dsa_refill_pool(const int32_t* miss_ids, const int32_t* miss_pos,
                          const int32_t* victim, const uint8_t* install,
                          const int32_t* miss_count, int B, int k, const void* sel_l,
                          void* pool_l, int P, int update_metadata, int32_t* pool_tags,
                          int32_t* fifo_ptr, const int32_t* ptr_next, int S, int W,
                          int32_t* err, cudaStream_t stream);

/* dsa_refill_pool_staged -- dsa_refill_pool for the staged layout: the rows
 * come from the pool's own staging rows, pool_l[b][victim[i]] =
 * pool_l[b][P + miss_pos[i]] (pool_l [B][P + k][576]; tags and pointers as
 * dsa_refill_pool's). Must run after this layer's sfa_mla_decode_pool, which
 * reads the slots read as hits in place. */
ts_status dsa_refill_pool_staged(const int32_t* miss_ids, const int32_t* miss_pos,
                                 const int32_t* victim, const uint8_t* install,
                                 const int32_t* miss_count, int B, int k, void* pool_l, int P,
                                 int update_metadata, int32_t* pool_tags, int32_t* fifo_ptr,
                                 const int32_t* ptr_next, int S, int W, int32_t* err,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * sfa_mla_decode -- sparse absorbed-MLA decode attention over the selection
 * ([GLM] §2.1 SFA; [TS] MLA section: one latent row is both K and V). For each
 * request b and head h, over the k selected rows K_j (576 values):
 *   s_j = scale * q[b][h] . K_j ;  p = softmax(s) ;
 *   out[b][h][:] = sum_j p_j K_j[0:512] ;  lse[b][h] = log(sum_j exp(s_j))
 * bf16 inputs, fp32 accumulation (tcgen05 tensor cores, TMEM accumulators),
 * the softmax weights rounded to bf16 for the second product, bf16 output.
 *
 *   q     bf16 [B][H][576]    16-byte aligned
 *   sel_l bf16 [B][k][576]    16-byte aligned
 *   out   bf16 [B][H][512]
 *   lse   float [B][H] or NULL
 *   ws    workspace of sfa_workspace_size(B, H, k) bytes, 256-byte aligned
 * A kernel wait that gives up sets TS_DEVERR_TIMEOUT.
 * ------------------------------------------------------------------------- */
size_t sfa_workspace_size(int B, int H, int k);
ts_status sfa_mla_decode(const void* q, const void* sel_l, int B, int H, int k,
                         float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                         int32_t* err, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * sfa_mla_decode_pool -- sfa_mla_decode whose rows come straight from a
 * staged-layout pool by the plan, with no selection buffer in between: the
 * gather fused into the attention ([GLM] §5 DsaServe's selection, consumed
 * where it lies; §2.1 SFA). Row j of request b is
 *   pool_l[b][src_map[b][j]]          for a hit (src_map >= 0),
 *   pool_l[b][P + first position of t] for a miss of t (src_map = -1 - t),
 * staged there by dsa_stage_misses. The tensor cores get the rows by TMA
 * gathers of four rows at a time. Same arithmetic, tile order and results
 * as sfa_mla_decode over the selection those rows make (bit for bit).
 *
 *   q        bf16 [B][H][576]
 *   pool_l   bf16 [B][P + k][576]     16-byte aligned; P + k <= 65536,
 *                                     B * (P + k) < 2^31
 *   src_map, miss_ids, miss_pos, miss_count, miss_rows   dsa_plan's
 *   out, lse, ws, ws_bytes            as sfa_mla_decode's
 * An out-of-range slot or a miss that is not in the miss list sets
 * TS_DEVERR_SLOT_RANGE / TS_DEVERR_ID_RANGE (that row then reads its own
 * staging row; the result is undefined). Must run after this layer's
 * dsa_stage_misses and before its dsa_refill_pool_staged.
 * ------------------------------------------------------------------------- */
ts_status sfa_mla_decode_pool(const void* q, const void* pool_l, int P, const int32_t* src_map,
                              const int32_t* miss_ids, const int32_t* miss_pos,
                              const int32_t* miss_count, const int32_t* miss_rows, int B, int H,
                              int k, float scale, void* out, float* lse, void* ws,
                              size_t ws_bytes, int32_t* err, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_group_step -- one decode step of an IndexShare group of `layers` layers,
 * enqueued by one call ([GLM] §5.1 model-side orchestration: one plan per
 * group, per-layer serve, refill on a side stream, metadata update at the
 * group's last layer; §4.4 SFA first, refill later). On the caller's three
 * streams it issues:
 *
 *   main   : ts_topk(scores) -> wait refilled -> dsa_plan -> signal planned
 *            -> wait for the previous step's output copies (host I/O only)
 *            -> for each layer l: wait gathered[l] -> sfa_mla_decode(l)
 *            (or on the layer streams below)
 *   gather : wait planned -> one launch gathering every layer (as
 *            dsa_gather_kv per layer, in layer order); the kernel itself
 *            writes gathered[l] once layer l's rows are all in
 *   side   : for each layer l: wait gathered[l] -> dsa_refill_pool(l) (the
 *            last layer also updates tags and FIFO pointers); then signal
 *            refilled
 *
 * Signals are writes of the step's sequence number into the caller's device
 * words `sync`: stream memory writes (cuStreamWriteValue32) for planned and
 * refilled, the gather kernel's own writes for gathered[l], and a one-thread
 * kernel's after each layer's attention (a stream memory write first takes a
 * system-wide memory barrier, slow while the gather keeps the host link
 * busy). Waits are
 * stream memory waits (cuStreamWaitValue32, compared wrap-around): the GPU's
 * front end polls device memory, with no event round trip, and no kernel
 * ever waits on another. Ordering: refill(l) evicts slots
 * gather(l) reads, so it waits for gather(l). The next step's plan reads the
 * tags the last refill writes, so it waits for `refilled`; the next step's
 * gather(l) rewrites sel[l], which sfa(l) and refill(l) of this step read: it
 * waits for the next plan, which follows every sfa on the main stream and
 * every refill. Every wait is enqueued after the signal it waits for, so
 * every wait ends.
 *
 * With layout = DSA_LAYOUT_STAGED the gather launch moves only the misses
 * (as dsa_stage_misses per layer), the attention is sfa_mla_decode_pool(l),
 * attended[l] is written after it on the main stream, and refill(l) waits for
 * attended[l] as well as gathered[l] (the attention reads the hit slots in
 * place; the refill overwrites some of them, from the staged rows).
 *
 * The descriptor holds the group's buffers (the caller owns all of them):
 *   ctx_len   int32 [B]                     k <= ctx_len[b] <= max_ctx
 *   pool      bf16  [layers][B][S*W][576]   the device pool of every layer
 *   pool_tags int32 [B][S*W], fifo_ptr int32 [B][S]   pool metadata
 *   host_kv   bf16  [layers][B][ctx_stride][576]  device-accessible address
 *                                           of pinned host memory
 *   ids ... ptr_next                        plan buffers, as dsa_plan's
 *   sel       bf16  [layers][B][k][576]     selection buffers
 *   out       bf16  [layers][B][H][512], lse float [layers][B][H] (or NULL)
 *   topk_ws / sfa_ws                        workspaces of ts_topk and
 *                                           sfa_mla_decode (sizes as theirs)
 *   err       int32 device error word (or NULL)
 *   sync      uint32 [5 + 3 * layers] device words, zero before the first step
 *             and touched by nothing else; step = 0 before the first step.
 *             Each call uses sequence number step + 1 and stores it in
 *             `step` (with the reuse policy it also swaps the buffers named
 *             below; no other field is written).
 * Step inputs: scores float [B][ctx_stride] (device); q bf16
 * [layers][B][H][576] (device); ids int32 [B][k] (device) or NULL -- when
 * given, the top-k is skipped and these ids are planned.
 * timing: NULL, or 2 * (3 + 2 * layers) events created by the caller, filled
 * as (start, end) pairs recorded on the launching stream around every
 * launch, in the order top-k, plan, gather (all layers), sfa[0..layers),
 * refill[0..layers) (the top-k pair is left alone when ids are given); a
 * NULL entry is not recorded (each recorded event costs the stream a little
 * time, so a caller may time only the launches it needs).
 * Every operation's arguments are validated before anything is enqueued;
 * 1 <= layers <= TS_MAX_LAYERS. If a launch fails after the first one, every
 * sync word still receives this step's number, written on the side stream
 * after the work already enqueued on all three streams (so no later wait is
 * left without its signal, and none passes early), and TS_ERR_CUDA is
 * returned; synchronize the three streams before trusting any buffer of the
 * group again.
 * ------------------------------------------------------------------------- */
#define TS_MAX_LAYERS 16

typedef struct {
  int B, layers, k, S, W, H, max_ctx;
  int64_t ctx_stride;
  float scale;
  const int32_t* ctx_len;
  void* pool;
  int32_t* pool_tags;
  int32_t* fifo_ptr;
  const void* host_kv;
  int32_t* ids;
  int32_t* src_map;
  int32_t* miss_ids;
  int32_t* miss_pos;
  int32_t* victim;
  uint8_t* install;
  int32_t* miss_count;
  int32_t* miss_rows;
  int32_t* ptr_next;
  void* sel;
  void* out;
  float* lse;
  void* topk_ws;
  size_t topk_ws_bytes;
  void* sfa_ws;
  size_t sfa_ws_bytes;
  int32_t* err;
  cudaStream_t main_stream, gather_stream, side_stream;
  uint32_t* sync;
  uint32_t step;
  /* pool policy: DSA_POLICY_FIFO, the set-associative FIFO pool above; or
   * DSA_POLICY_REUSE, the base design's adjacent-step reuse (dsa_plan_reuse):
   * the device keeps only the previous step's selection, prev_sel
   * ([layers][B][k][576]) and its ids prev_ids ([B][k], -1 before the first
   * step); pool, pool_tags, fifo_ptr, victim, install and ptr_next are not
   * used, no refill runs, and each call then swaps ids <-> prev_ids and
   * sel <-> prev_sel in the descriptor (so after a step prev_ids and
   * prev_sel hold that step's ids and selection). Reuse needs the top-k
   * inside the step (ids == NULL). */
  int policy;
  int32_t* prev_ids;
  void* prev_sel;
  /* where the attention reads its rows: DSA_LAYOUT_SELECTION, the selection
   * buffers above (gathered there by dsa_gather_kv's kernel); or
   * DSA_LAYOUT_STAGED, straight from the pool: `pool` is then
   * [layers][B][S*W + k][576], each request's rows S*W .. S*W+k-1 staging the
   * step's missed rows at their first positions; only the misses cross into
   * HBM (dsa_stage_misses' kernel), the attention is sfa_mla_decode_pool's,
   * each layer's refill waits for that layer's attention (the hits it read
   * stay in place until then), and `sel` is not used. Not with the reuse
   * policy. */
  int layout;
  /* DSA_POLICY_LRU: the fully associative LRU pool of P = S*W entries per
   * request (dsa_plan_lru): lru_order int32 [B][P], the slots from least to
   * most recently used (the identity for a cold pool); fifo_ptr, ptr_next
   * are not used and no refill runs (every install is written by the gather
   * as its row arrives). */
  int32_t* lru_order;
  /* DSA_LAYOUT_STAGED only, optional: uint32 [layers * B + 3 + layers]
   * device words (zeroed by each step itself). When given (and B <= 1024,
   * layers * B < 65535), each layer's attention starts as soon as the gather
   * is running and each of its CTAs waits, inside the kernel, for its own
   * request's missed rows of that layer (the gather counts every stored row
   * into arrived[l * B + b]); words layers * B .. + 2 count the gather's CTAs
   * that started, hold the step number once all have, and flag a gather that
   * gave up; the last `layers` words count each layer's attention CTAs that
   * started. The attention of a request then overlaps the gather of the
   * requests after it, and only the last requests' attention follows the
   * gather's end. NULL: each layer's attention waits for the whole layer's
   * rows. */
  uint32_t* arrived;
  /* With `arrived`, optional: `layers` streams (none of them NULL), and
   * sfa_ws must then hold one workspace per layer, layers *
   * sfa_workspace_size(B, H, k) bytes. Where one layer's attention has at
   * most half as many CTAs as the GPU has SMs (ceil(k / 512) * ceil(H / 128)
   * * B of them: few requests), layer l's attention (its two launches and
   * its words) then runs on layer_streams[l], launched once every CTA of
   * layer l - 1's attention has started (the CTAs still reach the SMs in the
   * gather's layer-then-request order), so the layers' attention overlaps,
   * and the main stream waits for every layer's attention at the end of the
   * step. Otherwise, or NULL: every layer's attention on the main stream, one
   * after another. */
  cudaStream_t* layer_streams;
} dsa_group;

#define DSA_POLICY_FIFO 0
#define DSA_POLICY_REUSE 1
#define DSA_POLICY_LRU 2
#define DSA_LAYOUT_SELECTION 0
#define DSA_LAYOUT_STAGED 1

ts_status dsa_group_step(dsa_group* g, const float* scores, const void* q, const int32_t* ids,
                         cudaEvent_t* timing);

/* dsa_group_step_host -- the same step with its inputs and its output in
 * page-locked host memory (device-accessible addresses, e.g. from
 * ts_host_alloc); every copy is inside the step, done by the SMs (ts_copy):
 *   main : scores_h -> scores_d, then the step as dsa_group_step
 *   side : wait planned >= step (this step's plan) -> layer by layer,
 *          q_h[l] -> layer l of one half of q_d (chosen by the step's parity)
 *          -> write step * layers + l into the sync word after the gather's
 *          ticket; layer l's attention waits for that value
 *   side : after each layer's attention (and that layer's refill), the
 *          layer's output -> out_h (it also stays in the descriptor's `out`);
 *          the next step's first attention waits for every layer's copy
 * So the scores the top-k waits for cross the host link alone, the queries
 * cross beside the gather, each layer's attention waits only for its own
 * layer's queries, and each layer's output crosses while later layers are
 * still gathered. The staging half a step writes was last read by the
 * attention of the step before the previous one, which precedes this step's
 * plan on the main stream.
 *   scores_h float [B][ctx_stride], q_h bf16 [layers][B][H][576],
 *   out_h bf16 [layers][B][H][512]      host (device-accessible addresses)
 *   scores_d float [B][ctx_stride], q_d bf16 2 x [layers][B][H][576]
 *                                        device staging, caller-owned
 * All 16-byte aligned. The top-k always runs. Returns as dsa_group_step. */
ts_status dsa_group_step_host(dsa_group* g, const float* scores_h, const void* q_h, void* out_h,
                              float* scores_d, void* q_d, cudaEvent_t* timing);

#ifdef __cplusplus
}
#endif

#endif /* DSAKV_H */
