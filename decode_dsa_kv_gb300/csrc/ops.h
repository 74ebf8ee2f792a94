// Host-side halves of the library's operations, for callers inside the
// library that enqueue several of them: every *_check validates arguments
// exactly as the public call does (and enqueues nothing); every *_enqueue
// launches on already-validated arguments. The public call is check, then
// enqueue.
#pragma once

#include "dsakv.h"

namespace dsakv {

ts_status topk_check(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                     int max_ctx, int k, int32_t* ids, const void* ws, size_t ws_bytes);
ts_status topk_enqueue(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                       int max_ctx, int k, int32_t* ids, void* ws, int32_t* err,
                       cudaStream_t stream);

ts_status plan_check(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                     const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                     int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos, int32_t* victim,
                     uint8_t* install, int32_t* miss_count, int32_t* miss_rows,
                     int32_t* ptr_next);
ts_status plan_enqueue(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                       const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                       int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos, int32_t* victim,
                       uint8_t* install, int32_t* miss_count, int32_t* miss_rows,
                       int32_t* ptr_next, int32_t* err, cudaStream_t stream);

ts_status plan_reuse_check(const int32_t* ids, const int32_t* prev_ids, const int32_t* ctx_len,
                           int B, int k, int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                           int32_t* miss_count, int32_t* miss_rows);
ts_status plan_reuse_enqueue(const int32_t* ids, const int32_t* prev_ids, const int32_t* ctx_len,
                             int B, int k, int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                             int32_t* miss_count, int32_t* miss_rows, int32_t* err,
                             cudaStream_t stream);

ts_status plan_lru_check(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                         const int32_t* pool_tags, const int32_t* lru_order, int P,
                         int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                         int32_t* victim, uint8_t* install,
                         int32_t* miss_count, int32_t* miss_rows);
ts_status plan_lru_enqueue(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                           int32_t* pool_tags, int32_t* lru_order, int P, int32_t* src_map,
                           int32_t* miss_ids, int32_t* miss_pos, int32_t* victim,
                           uint8_t* install, int32_t* miss_count,
                           int32_t* miss_rows, int32_t* err, cudaStream_t stream);

ts_status gather_check(const int32_t* src_map, const int32_t* miss_ids, const int32_t* miss_pos,
                       const int32_t* miss_count, const int32_t* miss_rows, int B, int k,
                       const void* pool_l, int P, const void* host_l, int64_t ctx_stride,
                       const int32_t* ctx_len, void* sel_l);
// `layers` consecutive layers in one launch (layer l's pool, host rows and
// selection start l * *_layer_bytes after pool_l / host_l / sel_l). With
// `done` non-null the kernel writes seq into done[l] once layer l's rows are
// all written (count: `layers` device words, zero between launches; the
// kernel leaves them zero). With `ticket` too (one device word, zero between
// launches; the kernel leaves it zero) and B <= 1024, the misses are handed
// out to the warps dynamically, layer after layer. With `victim` and `install` (dsa_plan's) given,
// the misses with install code 1 are also written into their victim slots
// of the pool as they arrive (the refill then needs only min_install = 2).
// With `arrived` (staged, dynamic and gather_streams(B, layers) only: its
// first layers * B + 3 uint32 words, zero before the launch; the attention's
// per-layer start counts follow them) the kernel adds every
// stored row to arrived[l * B + b], counts its CTAs in word layers * B,
// writes seq into word layers * B + 1 once every CTA runs, and sets word
// layers * B + 2 if it gives up (sfa_pool_enqueue's `arrived` waits on these).
ts_status gather_enqueue(const int32_t* src_map, const int32_t* miss_ids, const int32_t* miss_pos,
                         const int32_t* miss_count, const int32_t* miss_rows, int B, int k,
                         const void* pool_l, int P, const void* host_l, int64_t ctx_stride,
                         const int32_t* ctx_len, void* sel_l, int32_t* err, cudaStream_t stream,
                         int layers, size_t pool_layer_bytes, size_t host_layer_bytes,
                         size_t sel_layer_bytes, uint32_t* done, uint32_t* count, uint32_t seq,
                         const int32_t* victim, const uint8_t* install, bool staged,
                         uint32_t* ticket, uint32_t* arrived);

// most requests whose miss-count prefix fits beside the gather's pipes (its
// dynamic hand-out)
constexpr int kMaxDynamicB = 1024;
// whether a group of B requests x `layers` layers can count arrivals per
// request (the dynamic hand-out, and 16-bit row tags layer * B + b)
inline bool gather_streams(int B, int layers) {
  return B <= kMaxDynamicB && int64_t(layers) * B < 0xFFFF;
}

// The staged layout: a layer's pool tensor is [B][P + k][576]; rows P .. P+k-1
// of a request hold the step's missed rows at their first positions, so the
// attention reads every row straight from the pool (sfa_pool_*). gather_enqueue
// with staged = true moves only the misses (src_map, miss_rows and sel_l
// unused) into those rows; refill_enqueue with staged = true copies from them.
ts_status stage_check(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* miss_count,
                      int B, int k, const void* pool_l, int P, const void* host_l,
                      int64_t ctx_stride, const int32_t* ctx_len);

ts_status refill_check(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* victim,
                       const uint8_t* install, const int32_t* miss_count, int B, int k,
                       const void* sel_l, void* pool_l, int P, int update_metadata,
                       int32_t* pool_tags, int32_t* fifo_ptr, const int32_t* ptr_next, int S,
                       int W);
// `layers` consecutive layers in one launch: layer l's selection and pool
// start l * sel_layer_bytes / l * pool_layer_bytes after sel_l / pool_l.
// Only installs with install >= min_install are written (1: all; 2: those the
// gather did not write on arrival).
ts_status refill_enqueue(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* victim,
                         const uint8_t* install, const int32_t* miss_count, int B, int k,
                         const void* sel_l, void* pool_l, int P, int update_metadata,
                         int32_t* pool_tags, int32_t* fifo_ptr, const int32_t* ptr_next, int S,
                         int W, int32_t* err, cudaStream_t stream, int layers,
                         size_t sel_layer_bytes, size_t pool_layer_bytes, int min_install,
                         bool staged);

ts_status sfa_check(const void* q, const void* sel_l, int B, int H, int k, float scale,
                    void* out, const void* ws, size_t ws_bytes);
ts_status sfa_enqueue(const void* q, const void* sel_l, int B, int H, int k, float scale,
                      void* out, float* lse, void* ws, int32_t* err, cudaStream_t stream);
// CTAs of one attention launch's chunk kernel (chunks x head tiles x requests).
uint32_t sfa_chunk_ctas(int B, int H, int k);
// The attention reading its rows straight from a staged-layout pool by the
// plan (hits: the slot; misses: the staged row at P + first position).
ts_status sfa_pool_check(const void* q, const void* pool_l, int P, const int32_t* src_map,
                         const int32_t* miss_ids, const int32_t* miss_pos,
                         const int32_t* miss_count, const int32_t* miss_rows, int B, int H, int k,
                         float scale, void* out, const void* ws, size_t ws_bytes);
ts_status sfa_pool_enqueue(const void* q, const void* pool_l, int P, const int32_t* src_map,
                           const int32_t* miss_ids, const int32_t* miss_pos,
                           const int32_t* miss_count, const int32_t* miss_rows, int B, int H,
                           int k, float scale, void* out, float* lse, void* ws, int32_t* err,
                           cudaStream_t stream, const uint32_t* arrived = nullptr,
                           const uint32_t* gather_failed = nullptr,
                           uint32_t* started = nullptr);

}  // namespace dsakv
