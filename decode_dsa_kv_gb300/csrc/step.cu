// dsa_group_step: one decode step of an IndexShare group enqueued from native
// code (GLM-5.2 shared-Indexer KV Cache Offload, §5.1 model-side
// orchestration and §4.4 SFA first, refill later). The order of operations,
// the cross-stream signals and their proof of termination are the ones the
// header states; every argument is checked before the first launch.
//
// Cross-stream ordering uses device words holding the step's sequence number:
// a signal is a stream memory write issued on the producing stream (it lands
// when the stream's prior work is complete), a one-thread kernel's write
// after a layer's attention, or, for the per-layer gather signals, a write by
// the gather kernel itself once a layer's rows are in; a wait is a stream
// memory wait that blocks the consuming stream until the word, compared
// wrap-around, has reached that number. No kernel waits on another (except
// the streamed attention's bounded wait for its request's rows): only the
// streams' front end polls the words, in HBM.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "ops.h"

namespace dsakv {
namespace {

constexpr size_t kRowBytes = DSA_ROW_BYTES;
enum : int { kPlanned = 0, kRefilled = 1, kGathered = 2 };

// The step's inputs and output in page-locked host memory (device-accessible
// addresses), with the device staging they cross into (dsa_group_step_host).
struct HostIo {
  const float* scores_h;
  const void* q_h;
  void* out_h;
  float* scores_d;
  void* q_d;  // two halves of [layers][B][H][576], used by step parity
};

template <typename T>
T* at(T* base, int l, size_t layer_bytes) {
  using Byte = typename std::conditional<std::is_const<T>::value, const char, char>::type;
  return reinterpret_cast<T*>(reinterpret_cast<Byte*>(base) + size_t(l) * layer_bytes);
}

struct Layers {
  size_t pool, host, sel, out, lse, q;
};

Layers layer_bytes(const dsa_group& g) {
  Layers s;
  const size_t P = size_t(g.S) * g.W;
  s.pool = size_t(g.B) * P * kRowBytes;
  s.host = size_t(g.B) * size_t(g.ctx_stride) * kRowBytes;
  s.sel = size_t(g.B) * g.k * kRowBytes;
  s.out = size_t(g.B) * g.H * DSA_DV * 2;
  s.lse = size_t(g.B) * g.H * 4;
  s.q = size_t(g.B) * g.H * kRowBytes;
  return s;
}

using MemOpFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct MemOps {
  MemOpFn wait = nullptr, write = nullptr;
  bool ok = false;
};

const MemOps& memops() {
  static MemOps m = [] {
    MemOps r;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      r.wait = reinterpret_cast<MemOpFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      r.write = reinterpret_cast<MemOpFn>(p);
    r.ok = r.wait && r.write;
    return r;
  }();
  return m;
}

bool signal(cudaStream_t s, uint32_t* word, uint32_t v) {
  return memops().write(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(word), v,
                        CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
}

bool wait_for(cudaStream_t s, const uint32_t* word, uint32_t v) {
  return memops().wait(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(word), v,
                       CU_STREAM_WAIT_VALUE_GEQ) == CUDA_SUCCESS;
}

// One thread writes a layer's words once the stream's earlier kernels are
// complete (their writes are then visible on the GPU). A stream memory write
// does the same but first takes a system-wide memory barrier, which waits
// tens of microseconds while the gather keeps the host link busy (measured on
// GB300 at the large_batch shape: the two writes between two layers' attention
// launches held the next launch back by ~60 us; 18 us at decode_batch); a
// kernel's own stores need no such barrier.
__global__ void post_kernel(uint32_t* a, uint32_t va, uint32_t* b, uint32_t vb) {
  __threadfence();
  atomicExch(a, va);
  if (b) atomicExch(b, vb);
}

bool post(cudaStream_t s, uint32_t* a, uint32_t va, uint32_t* b = nullptr, uint32_t vb = 0) {
  post_kernel<<<1, 1, 0, s>>>(a, va, b, vb);
  return launch_status() == TS_OK;
}

}  // namespace
}  // namespace dsakv

using namespace dsakv;

namespace {

ts_status enqueue_step(dsa_group* gp, const float* scores, const void* q, const int32_t* ids,
                       cudaEvent_t* timing, const HostIo* io) {
  if (!gp || !q) return TS_ERR_INVALID_ARG;
  dsa_group& g = *gp;
  const int L = g.layers;
  if (L <= 0 || L > TS_MAX_LAYERS) return TS_ERR_INVALID_ARG;
  if (!ids && !scores) return TS_ERR_INVALID_ARG;
  const bool reuse = g.policy == DSA_POLICY_REUSE;
  const bool lru = g.policy == DSA_POLICY_LRU;
  if (!reuse && !lru && g.policy != DSA_POLICY_FIFO) return TS_ERR_INVALID_ARG;
  const bool refills = !reuse && !lru;  // only the FIFO pool defers installs
  const bool staged = g.layout == DSA_LAYOUT_STAGED;
  if (!staged && g.layout != DSA_LAYOUT_SELECTION) return TS_ERR_INVALID_ARG;
  if (staged && reuse) return TS_ERR_UNSUPPORTED;
  if (reuse && (ids || !g.prev_ids || !g.prev_sel)) return TS_ERR_INVALID_ARG;
  if (g.S <= 0 || g.W <= 0 || int64_t(g.S) * g.W > (1 << 24)) return TS_ERR_INVALID_ARG;
  if (!g.sync || (reinterpret_cast<uintptr_t>(g.sync) & 3u) != 0) return TS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(g.arrived) & 3u) != 0) return TS_ERR_INVALID_ARG;
  if (!aligned16(q)) return TS_ERR_INVALID_ARG;
  // streamed attention: each layer's attention CTAs wait inside the kernel
  // for their own request's staged rows, counted by the running gather
  const bool streamed = staged && g.arrived && gather_streams(g.B, L);
  // streamed, with layer streams: layer l's attention on its own stream, with
  // its own workspace (sfa_workspace_size each), where one layer's attention
  // CTAs fill at most half of the SMs. Measured on GB300 (streams against one
  // stream): long_context 0.189 against 0.292 ms a step, adversarial 0.343
  // against 0.374; at large_batch, whose every layer fills the SMs several
  // times over, the later layers' waiting CTAs held the SMs the refills
  // needed, and the step took 1.579 against 1.546 ms
  const size_t ws_layer = sfa_workspace_size(g.B, g.H, g.k);
  if (streamed && g.layer_streams) {
    for (int l = 0; l < L; ++l)
      if (!g.layer_streams[l]) return TS_ERR_INVALID_ARG;
    if (g.sfa_ws_bytes < size_t(L) * ws_layer) return TS_ERR_WORKSPACE;
  }
  const bool lanes = streamed && g.layer_streams &&
                     2 * int64_t(sfa_chunk_ctas(g.B, g.H, g.k)) <= int64_t(sm_count());
  // with reuse, the "pool" is the previous step's selection: k rows per request
  const int P = reuse ? g.k : g.S * g.W;
  Layers lb = layer_bytes(g);
  if (reuse) lb.pool = lb.sel;
  if (staged) lb.pool = size_t(g.B) * (size_t(P) + g.k) * kRowBytes;
  const void* pool = reuse ? static_cast<const void*>(g.prev_sel) : g.pool;
  const int32_t* plan_ids = ids ? ids : g.ids;

  // every operation's host checks first (layer 0 stands for all layers: the
  // layer strides are whole multiples of 16 bytes)
  ts_status st = TS_OK;
  if (!ids)
    st = topk_check(scores, g.ctx_stride, g.ctx_len, g.B, g.max_ctx, g.k, g.ids, g.topk_ws,
                    g.topk_ws_bytes);
  if (st == TS_OK)
    st = reuse ? plan_reuse_check(plan_ids, g.prev_ids, g.ctx_len, g.B, g.k, g.src_map, g.miss_ids,
                                  g.miss_pos, g.miss_count, g.miss_rows)
         : lru ? plan_lru_check(plan_ids, g.ctx_len, g.B, g.k, g.pool_tags, g.lru_order, P,
                                g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install,
                                g.miss_count, g.miss_rows)
               : plan_check(plan_ids, g.ctx_len, g.B, g.k, g.pool_tags, g.fifo_ptr, g.S, g.W,
                            g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install, g.miss_count,
                            g.miss_rows, g.ptr_next);
  if (st == TS_OK)
    st = staged ? stage_check(g.miss_ids, g.miss_pos, g.miss_count, g.B, g.k, g.pool, P, g.host_kv,
                              g.ctx_stride, g.ctx_len)
                : gather_check(g.src_map, g.miss_ids, g.miss_pos, g.miss_count, g.miss_rows, g.B,
                               g.k, pool, P, g.host_kv, g.ctx_stride, g.ctx_len, g.sel);
  if (st == TS_OK && refills)
    st = refill_check(g.miss_ids, g.miss_pos, g.victim, g.install, g.miss_count, g.B, g.k,
                      staged ? g.pool : g.sel, g.pool, P, 1, g.pool_tags, g.fifo_ptr, g.ptr_next,
                      g.S, g.W);
  if (st == TS_OK)
    st = staged ? sfa_pool_check(q, g.pool, P, g.src_map, g.miss_ids, g.miss_pos, g.miss_count,
                                 g.miss_rows, g.B, g.H, g.k, g.scale, g.out, g.sfa_ws,
                                 g.sfa_ws_bytes)
                : sfa_check(q, g.sel, g.B, g.H, g.k, g.scale, g.out, g.sfa_ws, g.sfa_ws_bytes);
  if (st != TS_OK) return st;
  if (!memops().ok) return TS_ERR_UNSUPPORTED;

  const uint32_t seq = g.step + 1;
  g.step = seq;
  cudaStream_t m = g.main_stream, gs = g.gather_stream, side = g.side_stream;
  uint32_t* planned = g.sync + kPlanned;
  uint32_t* refilled = g.sync + kRefilled;
  uint32_t* gathered = g.sync + kGathered;
  uint32_t* counts = g.sync + kGathered + L;  // the gather's per-layer warp counts
  uint32_t* attended = g.sync + kGathered + 2 * L;  // staged layout: a layer's attention is done
  uint32_t* ticket = g.sync + kGathered + 3 * L;    // the gather's miss hand-out
  uint32_t* qcopied = ticket + 1;                   // host I/O: the queries are in
  uint32_t* outcopied = ticket + 2;                 // host I/O: a layer's output is out
  // streamed: per (layer, request) arrival counts, then the gather's started
  // CTAs, the started flag and the gave-up flag
  uint32_t* started = streamed ? g.arrived + size_t(L) * g.B + 1 : nullptr;
  uint32_t* gave_up = streamed ? started + 1 : nullptr;
  // streamed: per layer, the attention CTAs that have started
  uint32_t* lstarted = streamed ? g.arrived + size_t(L) * g.B + 3 : nullptr;
  const uint32_t nctas = sfa_chunk_ctas(g.B, g.H, g.k);
  auto astream = [&](int l) { return lanes ? g.layer_streams[l] : m; };

  // with host I/O: the copies' sizes; this step's half of the query staging
  const size_t scores_bytes = size_t(g.B) * size_t(g.ctx_stride) * 4;
  const size_t q_bytes = size_t(L) * lb.q;
  void* q_stage = io ? static_cast<char*>(io->q_d) + (seq & 1u) * q_bytes : nullptr;
  if (io) q = q_stage;
  // (a NULL entry of `timing` is left out: a caller may time only some launches)
  auto rec = [&](int slot, int end, cudaStream_t s) {
    cudaEvent_t e = timing ? timing[2 * slot + end] : nullptr;
    return e ? cudaEventRecord(e, s) == cudaSuccess : true;
  };

  bool ok = true;
  // streamed: the counts start from zero, ahead of the top-k (the previous
  // step's attention, their last reader, ran earlier on this stream, and
  // every count it waited for was complete; this step's gather waits for the
  // plan, after this)
  if (streamed)
    ok = cudaMemsetAsync(g.arrived, 0, (size_t(L) * g.B + 3 + L) * 4, m) == cudaSuccess;
  // with host I/O the scores cross first, on the main stream ahead of the top-k
  if (io) ok = ok && ts_copy(io->scores_d, io->scores_h, scores_bytes, m) == TS_OK;
  if (!ids) {
    ok = ok && rec(0, 0, m) &&
         topk_enqueue(scores, g.ctx_stride, g.ctx_len, g.B, g.max_ctx, g.k, g.ids, g.topk_ws,
                      g.err, m) == TS_OK &&
         rec(0, 1, m);
  }
  ok = ok && wait_for(m, refilled, seq - 1) && rec(1, 0, m) &&
       (reuse ? plan_reuse_enqueue(plan_ids, g.prev_ids, g.ctx_len, g.B, g.k, g.src_map,
                                   g.miss_ids, g.miss_pos, g.miss_count, g.miss_rows, g.err, m)
        : lru ? plan_lru_enqueue(plan_ids, g.ctx_len, g.B, g.k, g.pool_tags, g.lru_order, P,
                                 g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install,
                                 g.miss_count, g.miss_rows, g.err, m)
              : plan_enqueue(plan_ids, g.ctx_len, g.B, g.k, g.pool_tags, g.fifo_ptr, g.S, g.W,
                             g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install,
                             g.miss_count, g.miss_rows, g.ptr_next, g.err, m)) == TS_OK &&
       rec(1, 1, m) && signal(m, planned, seq) && wait_for(gs, planned, seq);
  // every attention of this step overwrites `out`: with host I/O in the step
  // before, the side stream copied each layer of it out, and the last copy
  // wrote (seq - 1) * L + L - 1 (without, the step wrote that itself). One
  // wait here, on the main stream ahead of the gather's traffic, covers
  // every layer
  // (with layer streams each layer's stream waits for its own layer's copy)
  const uint32_t seqL = seq * uint32_t(L);
  ok = ok && (lanes || seq == 1 || wait_for(m, outcopied, seqL - 1));
  // one launch gathers every layer and writes seq into gathered[l] from the
  // device as soon as layer l's rows are in (no ramp between layers); it also
  // installs the misses whose victim slots no hit of the step reads (install
  // code 1), so each layer's refill copies only the code-2 rows
  ok = ok && rec(2, 0, gs) &&
       gather_enqueue(g.src_map, g.miss_ids, g.miss_pos, g.miss_count, g.miss_rows, g.B, g.k, pool,
                      P, g.host_kv, g.ctx_stride, g.ctx_len, g.sel, g.err, gs, L, lb.pool,
                      lb.host, lb.sel, gathered, counts, seq, reuse ? nullptr : g.victim,
                      reuse ? nullptr : g.install, staged, ticket,
                      streamed ? g.arrived : nullptr) == TS_OK &&
       rec(2, 1, gs);
  // with host I/O the queries cross on the side stream once this step's plan
  // is done (the scores the top-k waits for then cross the host link alone),
  // into this step's staging half; that half's last reader, the attention of
  // step seq - 2, came before planned >= seq - 1 on the main stream (the
  // signal is enqueued already, so the wait ends). Layer by layer, each copy
  // followed by the word's next value seq * L + l, which layer l's attention
  // waits for (values grow step after step)
  if (io) {
    ok = ok && wait_for(side, planned, seq);
    for (int l = 0; ok && l < L; ++l)
      ok = ts_copy(at(q_stage, l, lb.q), at(io->q_h, l, lb.q), lb.q, side) == TS_OK &&
           post(side, qcopied, seq * uint32_t(L) + l);
  }
  // per layer: the attention on the main stream, the refill beside it on the
  // side stream; the last refill also updates the metadata. The staged
  // attention reads hit rows from the pool itself, so the layer's refill
  // (which overwrites slots read as hits) waits for that attention
  // Streamed, the first layer's attention launches once every gather CTA
  // runs (so the gather that its CTAs wait for never waits for SMs they
  // hold) and the later layers follow it on the stream.
  // With layer streams, layer l's attention runs on layer_streams[l] and
  // launches once every CTA of layer l - 1's attention has started, so the
  // CTAs still reach the SMs in the gather's layer-then-request order (no
  // waiting CTA of a later layer takes an SM a CTA of an earlier layer
  // needs) while the layers overlap where one layer's CTAs leave SMs idle;
  // every layer stream first waits for this step's gather to run (after the
  // counts were zeroed), and for the step before's copy of its layer's output.
  // Each layer's output crosses to the host (host I/O) on the side stream,
  // after the layer's refill; outcopied then holds seq * L + l (a step
  // without host I/O writes the value itself: with attended[l], or with
  // layer streams once on the main stream after every layer). Between two
  // layers' attention launches a stream holds only kernels: the words are
  // written by post_kernel, not by stream memory writes.
  for (int l = 0; ok && l < L; ++l) {
    float* lse_l = g.lse ? at(g.lse, l, lb.lse) : nullptr;
    const cudaStream_t a = astream(l);
    void* ws_l = lanes ? static_cast<char*>(g.sfa_ws) + size_t(l) * ws_layer : g.sfa_ws;
    ok = (streamed ? ((l > 0 && !lanes) || wait_for(a, started, seq))
                   : wait_for(a, gathered + l, seq)) &&
         (!lanes || l == 0 || wait_for(a, lstarted + l - 1, nctas)) &&
         (!lanes || seq == 1 || wait_for(a, outcopied, seqL - L + l)) &&
         (!io || wait_for(a, qcopied, seqL + l)) && rec(3 + l, 0, a) &&
         (staged ? sfa_pool_enqueue(at(q, l, lb.q), at(g.pool, l, lb.pool), P, g.src_map,
                                    g.miss_ids, g.miss_pos, g.miss_count, g.miss_rows, g.B, g.H,
                                    g.k, g.scale, at(g.out, l, lb.out), lse_l, ws_l, g.err, a,
                                    streamed ? g.arrived + size_t(l) * g.B : nullptr, gave_up,
                                    streamed ? lstarted + l : nullptr)
                 : sfa_enqueue(at(q, l, lb.q), at(g.sel, l, lb.sel), g.B, g.H, g.k, g.scale,
                               at(g.out, l, lb.out), lse_l, g.sfa_ws, g.err, a)) == TS_OK &&
         rec(3 + l, 1, a) &&
         post(a, attended + l, seq, (io || lanes) ? nullptr : outcopied, seqL + l);
    // (staged: the refill copies staged rows into victim slots; an attention
    // ends after its requests' rows are in unless its wait for them ran out,
    // so the refill also waits for the gather's layer)
    if (refills)
      ok = ok && wait_for(side, (staged ? attended : gathered) + l, seq) &&
           (!staged || wait_for(side, gathered + l, seq)) && rec(3 + L + l, 0, side) &&
           refill_enqueue(g.miss_ids, g.miss_pos, g.victim, g.install, g.miss_count, g.B, g.k,
                          staged ? nullptr : at(g.sel, l, lb.sel), at(g.pool, l, lb.pool), P,
                          l == L - 1, g.pool_tags, g.fifo_ptr, g.ptr_next, g.S, g.W, g.err, side,
                          1, lb.sel, lb.pool, 2, staged) == TS_OK &&
           rec(3 + L + l, 1, side) &&
           // the next plan waits for the last refill, not for the last copy
           (l < L - 1 || signal(side, refilled, seq));
    if (io)
      ok = ok && wait_for(side, attended + l, seq) &&
           ts_copy(at(io->out_h, l, lb.out), at(g.out, l, lb.out), lb.out, side) == TS_OK &&
           post(side, outcopied, seqL + l);
  }
  // with layer streams the main stream then waits for every layer's
  // attention: what follows on it (the next step's plan, which the next
  // gather waits for) comes after every attention of this step
  if (lanes) {
    for (int l = 0; ok && l < L; ++l) ok = wait_for(m, attended + l, seq);
    ok = ok && (io || post(m, outcopied, seqL + L - 1));
  }
  if (lru) {
    // no refill: the plan updated the pool's metadata and the gather wrote
    // every install as its row arrived. The next plan only has to follow
    // this step's (it does, on the main stream); the next gather, which
    // installs into slots this step's attention may read (staged layout),
    // waits for the next plan, after this step's last attention
    ok = ok && signal(m, refilled, seq);
  } else if (reuse) {
    // no refill: this step's selection and ids become the next step's
    // "pool". The next step's top-k writes the old previous ids, which this
    // step's plan read (earlier on the main stream); its gather writes the old
    // previous selection, which this step's gather read (it waits for the
    // next plan, after this step's attention, after this gather's last layer)
    ok = ok && signal(m, refilled, seq);
    if (ok) {
      int32_t* t_ids = g.ids;
      g.ids = g.prev_ids;
      g.prev_ids = t_ids;
      void* t_sel = g.sel;
      g.sel = g.prev_sel;
      g.prev_sel = t_sel;
    }
  }
  if (!ok) {
    // give every signal word this step's number, so that no wait enqueued
    // now or by the next call is left without its signal. The side stream
    // first waits for everything already enqueued on the other streams
    // (every wait enqueued there has its signal: a per-layer wait is
    // enqueued only after the launch that writes it), so no signal lands
    // while a kernel of this step still reads or writes the pool
    cudaEvent_t ev[2 + TS_MAX_LAYERS] = {};
    cudaStream_t others[2 + TS_MAX_LAYERS] = {m, gs};
    const int n_others = 2 + (lanes ? L : 0);
    for (int l = 0; lanes && l < L; ++l) others[2 + l] = g.layer_streams[l];
    for (int i = 0; i < n_others; ++i)
      if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess &&
          cudaEventRecord(ev[i], others[i]) == cudaSuccess)
        cudaStreamWaitEvent(side, ev[i], 0);
    for (int i = 0; i < kGathered + L; ++i) signal(side, g.sync + i, seq);
    for (int i = 0; i < L; ++i) signal(side, attended + i, seq);
    if (streamed) {  // and no attention CTA keeps waiting for rows
      signal(side, started, seq);
      signal(side, gave_up, seq);
    }
    if (io) signal(side, qcopied, seqL + L - 1);
    signal(side, outcopied, seqL + L - 1);
    for (int i = 0; i < n_others; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  return TS_OK;
}

}  // namespace

extern "C" ts_status dsa_group_step(dsa_group* gp, const float* scores, const void* q,
                                    const int32_t* ids, cudaEvent_t* timing) {
  return enqueue_step(gp, scores, q, ids, timing, nullptr);
}

extern "C" ts_status dsa_group_step_host(dsa_group* gp, const float* scores_h, const void* q_h,
                                         void* out_h, float* scores_d, void* q_d,
                                         cudaEvent_t* timing) {
  if (!gp || !scores_h || !q_h || !out_h || !scores_d || !q_d) return TS_ERR_INVALID_ARG;
  if (!aligned16(scores_h) || !aligned16(q_h) || !aligned16(out_h) || !aligned16(scores_d) ||
      !aligned16(q_d))
    return TS_ERR_INVALID_ARG;
  const HostIo io{scores_h, q_h, out_h, scores_d, q_d};
  return enqueue_step(gp, scores_d, q_d, nullptr, timing, &io);
}
