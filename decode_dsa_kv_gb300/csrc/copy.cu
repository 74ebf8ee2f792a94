// Row movement of the decode-step KV path: dsa_gather_kv serves one layer's
// selected rows (GLM-5.2 shared-Indexer KV Cache Offload, §5 DsaServe and
// §5.1; the base design's GatherSelectionKvCache, §2.1), dsa_refill_pool
// installs one layer's missed rows into their FIFO victim slots and, at the
// group's last layer, updates the pool metadata (§4.4 refill after SFA, §5
// DsaInstall, §5.1 metadata update at the group's last layer).
//
// Both are pure copies of 1152-byte rows: HBM for pool hits, pinned host
// memory read in place over the host link for misses. The gather moves rows
// through shared memory with bulk async copies, so a few SMs keep enough rows
// in flight for the link and for HBM, and the attention keeps the rest.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "ops.h"

namespace dsakv {
namespace {

constexpr int kMissCtas = 8;  // gather CTAs reading missed rows over the host link
constexpr int kHitCtas = 16;  // gather CTAs copying the other positions

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(uint4* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Rows through shared memory with bulk async copies (no registers hold the
// rows, so a few SMs keep enough rows in flight for the host link or HBM).
// Lane 0 of a warp issues everything: a row is loaded into one of
// kPipeSlots ring slots and stored from there once it has arrived; a slot is
// loaded again only after the store that read it kPipeLag stores earlier is
// done reading. Waits are bounded; after a timeout the pipe issues nothing
// more, still waits (bounded) for every load in flight, and reports.
constexpr int kPipeSlots = 12;
constexpr int kPipeLag = 2;
constexpr int kPipeAhead = kPipeSlots - kPipeLag;  // loads in flight per warp
constexpr int kPipeRetire = 4;  // stores after a layer's last before it counts out
constexpr int kPipeWarps = 16;                     // warps per gather CTA
constexpr uint64_t kBulkWaitNs = 100000000ull;     // 100 ms
constexpr int kTagRing = 48;  // pushed rows' request tags, by row number (see RowPipe::publish)
constexpr int kNoTag = 0xFFFF;  // a row counted into no request's arrivals
// A warp's shared memory: the ring, its barriers, the rows' targets, the
// rows' tags, then the words it shares with the CTA's counting warp.
constexpr size_t kPipeTagOffset = kPipeSlots * (DSA_ROW_BYTES + 24);
constexpr size_t kPipeWordsOffset = kPipeTagOffset + kTagRing * 2;
constexpr size_t kPipeWarpBytes = kPipeWordsOffset + 16;
constexpr uint64_t kCountIdleNs = 1000000000ull;  // the counting warp gives up after 1 s idle
constexpr size_t kPipeSmemBytes = kPipeWarps * kPipeWarpBytes;
// misses per ticket: a layer's completion waits for the last batch of it any
// warp took, so smaller batches let the layers finish closer to their share
constexpr int kTicketRows = 16;
// (the kernel's static shared memory, the scan scratch and what the compiler
// adds, is counted as 256 bytes)
static_assert(kPipeSmemBytes + (kMaxDynamicB + 1) * 4 + 256 <= 227 * 1024, "shared memory");
static_assert(kPipeWarpBytes % 16 == 0, "rings start on 16-byte boundaries");
constexpr int kGatherThreads = (kPipeWarps + 1) * 32;  // the pipes and the counting warp

// Words a pipe warp shares with its CTA's counting warp (streamed attention):
// rows [0, published) of the warp are stored, rows [0, consumed) are counted,
// finished once the warp has published its last row.
struct PipeWords {
  uint32_t published, consumed, finished, pad;
};
__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

struct RowPipe {
  uint8_t* ring;
  uint64_t* bars;
  uint4** to;
  uint4** to2;  // a second target of the row, or null
  uint32_t issued, stored;
  bool failed;
  // layer completion: the warp counts itself out of layer `pend` (its rows
  // are the items below pend_end) once kPipeRetire later stores are issued,
  // after waiting for all but those; the pipe never drains between layers
  int pend;
  uint32_t pend_end;
  int nw;
  uint32_t *count, *done, seq;
  uint32_t* ticket;  // dynamic miss hand-out: reset by the last warp of the last layer
  int last;
  // per-request arrival counts (streamed attention): row i's counter index
  // (layer * B + request, or kNoTag) sits in tags[i % kTagRing] from its
  // push until the counting warp has read it; rows below `published` are
  // stored, which the warp tells the counting warp through `words`
  uint32_t* arrived;
  uint16_t* tags;
  PipeWords* words;
  uint32_t published, consumed;
  bool self_count;  // the warp releases and counts its rows itself (no counting warp)

  __device__ void init(uint8_t* warp_smem, int nw_, uint32_t* count_, uint32_t* done_,
                       uint32_t seq_, uint32_t* ticket_, int last_, uint32_t* arrived_,
                       bool self_count_) {
    ring = warp_smem;
    bars = reinterpret_cast<uint64_t*>(warp_smem + kPipeSlots * DSA_ROW_BYTES);
    to = reinterpret_cast<uint4**>(bars + kPipeSlots);
    to2 = to + kPipeSlots;
    issued = stored = 0;
    failed = false;
    pend = -1;
    pend_end = 0;
    nw = nw_;
    count = count_;
    done = done_;
    seq = seq_;
    ticket = ticket_;
    last = last_;
    arrived = arrived_;
    tags = reinterpret_cast<uint16_t*>(warp_smem + kPipeTagOffset);
    words = reinterpret_cast<PipeWords*>(warp_smem + kPipeWordsOffset);
    published = consumed = 0;
    self_count = self_count_;
    words->published = words->consumed = words->finished = 0;
    for (int s = 0; s < kPipeSlots; ++s) mbar_init(bars + s, 1);
    mbar_fence_init();
  }
  // The warp's rows of layer l are written: count it out (the last warp of
  // the launch writes seq into done[l]).
  __device__ void signal(int l) {
    if (!done) return;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    if (atomicAdd(count + l, 1u) == static_cast<uint32_t>(nw) - 1) {
      __threadfence();
      count[l] = 0;
      // every warp has taken its last ticket before counting out of the last layer
      if (ticket && l == last) *ticket = 0;
      atomicExch(done + l, seq);
    }
  }
  // Rows below n are stored (the caller waited for their store groups):
  // make them count. Either this thread releases them at GPU scope and adds
  // them to their requests' arrival counts itself (self_count), or it tells
  // the CTA's counting warp, which does (their bulk writes ordered before the
  // shared word by a CTA-scope release). A GPU-scope fence on an SM whose
  // warps keep host reads in flight waits microseconds (measured on GB300:
  // 7 us on average from a pipe thread at 128 x 32,768, 1.9 us at 32 x
  // 65,536, 30 us from a separate warp at 128 x 32,768); the pipes only
  // afford it when the launch has reads in flight to spare (see
  // gather_enqueue).
  __device__ void publish(uint32_t n) {
    if (!arrived || failed || n <= published) return;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    if (self_count) {
      __threadfence();
      int tag = tags[published % kTagRing];
      uint32_t run = 0;
      for (uint32_t i = published; i < n; ++i) {
        const int t = tags[i % kTagRing];
        if (t != tag) {
          if (tag != kNoTag) atomicAdd(arrived + tag, run);
          tag = t;
          run = 0;
        }
        ++run;
      }
      if (tag != kNoTag) atomicAdd(arrived + tag, run);
    } else {
      st_release_cta(&words->published, n);
    }
    published = n;
  }
  // Store the oldest row in flight (or, after a failure, only wait for it).
  __device__ void store_one() {
    const uint32_t i = stored++;
    const int s = static_cast<int>(i % kPipeSlots);
    const bool ok = mbar_wait_timed(bars + s, (i / kPipeSlots) & 1u, kBulkWaitNs);
    if (!ok) failed = true;
    if (ok && !failed) {
      bulk_store(to[s], ring + s * DSA_ROW_BYTES, DSA_ROW_BYTES);
      if (to2[s]) bulk_store(to2[s], ring + s * DSA_ROW_BYTES, DSA_ROW_BYTES);
      bulk_commit();
    }
    if (pend >= 0 && stored == pend_end + kPipeRetire) {
      // every store group but the last kPipeRetire (all after pend_end) done
      if (failed) bulk_wait_all();
      else bulk_wait<kPipeRetire>();
      publish(stored - kPipeRetire);
      signal(pend);
      pend = -1;
    } else if (arrived && (stored & 3u) == 0 && stored > kPipeRetire) {
      // every fourth store: the rows whose stores are done are published
      bulk_wait<kPipeRetire>();
      publish(stored - kPipeRetire);
    }
  }
  __device__ void push(const uint4* from, uint4* dst, uint4* dst2 = nullptr, int tag = kNoTag) {
    if (failed) return;
    while (stored + kPipeAhead <= issued) store_one();
    if (failed) return;
    if (arrived && !self_count && issued - consumed >= kTagRing) {
      // the tag entry this row takes is still to be read by the counting warp
      const uint64_t t0 = globaltimer_ns();
      while (issued - (consumed = ld_acquire_cta(&words->consumed)) >= kTagRing) {
        if (globaltimer_ns() - t0 > kBulkWaitNs) {
          failed = true;
          return;
        }
        __nanosleep(64);
      }
    }
    bulk_wait_read<kPipeLag>();
    const int s = static_cast<int>(issued % kPipeSlots);
    to[s] = dst;
    to2[s] = dst2;
    tags[issued % kTagRing] = static_cast<uint16_t>(tag);
    mbar_expect_tx(bars + s, DSA_ROW_BYTES);
    bulk_load(ring + s * DSA_ROW_BYTES, from, DSA_ROW_BYTES, bars + s);
    ++issued;
  }
  // Every row of layer l is pushed. A layer still pending from before is
  // completed first (it had fewer than kPipeRetire stores after it).
  __device__ void end_layer(int l) {
    if (pend >= 0) {
      while (stored < issued) store_one();
      if (pend >= 0) {
        bulk_wait_all();
        publish(stored);
        signal(pend);
      }
    }
    pend = l;
    pend_end = issued;
  }
  // Every row pushed stored and written; the pending layer counted out.
  __device__ void finish() {
    while (stored < issued) store_one();
    bulk_wait_all();
    publish(stored);
    if (arrived && !self_count) st_release_cta(&words->finished, 1u);
    if (pend >= 0) signal(pend);
    pend = -1;
  }
};

// The counting warp of a streamed gather CTA: lane w follows pipe warp w's
// published rows and adds them to their requests' arrival counts, one
// atomic per run of rows of one request, after a GPU-scope fence (the rows'
// writes, ordered before `published`, become visible to the attention before
// the counts). The lanes sweep together, so a sweep with new rows in any pipe
// costs one fence for the warp (on an SM whose pipes keep host reads in
// flight a fence takes microseconds; one per lane and sweep fell behind the
// pipes at the large_batch shape). Gives up after kCountIdleNs without progress.
__device__ void count_arrivals(uint8_t* smem, uint32_t* arrived, uint32_t* gave_up, int lane) {
  const bool mine = lane < kPipeWarps;
  uint8_t* base = smem + size_t(mine ? lane : 0) * kPipeWarpBytes;
  const uint16_t* tags = reinterpret_cast<const uint16_t*>(base + kPipeTagOffset);
  PipeWords* words = reinterpret_cast<PipeWords*>(base + kPipeWordsOffset);
  uint32_t seen = 0;
  bool done = !mine;
  uint64_t t_idle = globaltimer_ns();
  for (;;) {
    uint32_t fin = 1, p = seen;
    if (!done) {
      fin = ld_acquire_cta(&words->finished);  // (read first: p is then the last value)
      p = ld_acquire_cta(&words->published);
    }
    const bool work = p > seen;
    if (__any_sync(0xffffffffu, work)) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      if (work) {
        int tag = tags[seen % kTagRing];
        uint32_t run = 0;
        for (uint32_t i = seen; i < p; ++i) {
          const int t = tags[i % kTagRing];
          if (t != tag) {
            if (tag != kNoTag) atomicAdd(arrived + tag, run);
            tag = t;
            run = 0;
          }
          ++run;
        }
        if (tag != kNoTag) atomicAdd(arrived + tag, run);
        seen = p;
        st_release_cta(&words->consumed, seen);
      }
      t_idle = globaltimer_ns();
    } else {
      if (fin) done = true;
      if (__all_sync(0xffffffffu, done)) break;
      // (lane 0's clock decides for the warp, which leaves the loop together)
      if (__shfl_sync(0xffffffffu, globaltimer_ns() - t_idle > kCountIdleNs ? 1 : 0, 0)) {
        if (lane == 0) atomicExch(gave_up, 1u);  // the attention stops waiting for these counts
        break;
      }
      __nanosleep(128);
    }
  }
}

// Row lists of one layer (see gather_kernel).
struct GatherLayer {
  uint4* pool;  // read for hits; written for installs on arrival
  const uint4* host;
  uint4* sel;
};

// Source and targets of miss i of request b (the plan's miss list): the host
// row, its place in the selection (or staging rows), and, for an install with
// code 1, its victim slot. False (with bits in `bad`) for a corrupt entry.
__device__ __forceinline__ bool miss_targets(const GatherLayer& L, const int32_t* miss_ids,
                                             const int32_t* miss_pos, const int32_t* victim,
                                             const uint8_t* install, int b, int i, int k, int P,
                                             int sel_rows, int pool_rows, int64_t ctx_stride,
                                             const int32_t* ctx_len, const uint4*& from,
                                             uint4*& to, uint4*& to2, int& bad) {
  const bool in = i >= 0 && i < k;  // (a count past k is corrupt)
  const int64_t s = int64_t(b) * k + i;
  const int t = in ? __ldg(miss_ids + s) : -1;
  const int j = in ? __ldg(miss_pos + s) : -1;
  if (t < 0 || t >= __ldg(ctx_len + b) || t >= ctx_stride || j < 0 || j >= k) {
    bad |= TS_DEVERR_ID_RANGE;
    return false;
  }
  from = L.host + (int64_t(b) * ctx_stride + t) * DSA_ROW_CHUNKS;
  to = L.sel + (int64_t(b) * sel_rows + j) * DSA_ROW_CHUNKS;
  to2 = nullptr;
  if (victim && __ldg(install + s) == 1) {
    const int v = __ldg(victim + s);
    if (v >= 0 && v < P) to2 = L.pool + (int64_t(b) * pool_rows + v) * DSA_ROW_CHUNKS;
    else bad |= TS_DEVERR_SLOT_RANGE;
  }
  return true;
}

// Lane 0 pushes the rows of the lanes in `mask` through the warp's pipe.
__device__ __forceinline__ void push_lanes(uint32_t mask, const uint4* from, uint4* to, uint4* to2,
                                           int lane, RowPipe& pipe, int tag = kNoTag) {
  while (mask) {
    const int q = __ffs(mask) - 1;
    mask &= mask - 1;
    const uint4* f = reinterpret_cast<const uint4*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(from), q));
    uint4* t = reinterpret_cast<uint4*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(to), q));
    uint4* t2 =
        reinterpret_cast<uint4*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(to2), q));
    const int tg = __shfl_sync(0xffffffffu, tag, q);
    if (lane == 0) pipe.push(f, t, t2, tg);
    __syncwarp();
  }
}

// The misses of all requests, concatenated: the warp takes miss indices
// m = w, w + nrole, ... (request b holds miss_count[b] of them), so every miss
// warp gets the same number of host rows whatever the spread of misses over
// requests. Looked up 32 at a time, one candidate per lane; `mask` holds the
// lanes with a row to move, which lane 0 pushes through the warp's pipe.
// With `victim` given, a miss with install code 1 (its victim slot is read by
// no position of this step) is also written into that slot of the pool as it
// arrives, which leaves the refill only the code-2 installs.
__device__ __forceinline__ void gather_misses(const GatherLayer& L, const int32_t* miss_ids,
                                              const int32_t* miss_pos, const int32_t* miss_count,
                                              const int32_t* victim, const uint8_t* install,
                                              int B, int k, int P, int sel_rows, int pool_rows,
                                              int64_t ctx_stride, const int32_t* ctx_len, int w,
                                              int nrole, int lane, RowPipe& pipe, int& bad) {
  // indices below B * k < 2^31 (B <= 65535, k <= 8192) fit in 32 bits
  const uint4* host = L.host;
  uint4* sel = L.sel;
  int m1 = w, base1 = 0;
  int b1 = 0, cnt1 = __ldg(miss_count);
  uint32_t mask = 0;
  const uint4* my_from = nullptr;
  uint4* my_to = nullptr;
  uint4* my_to2 = nullptr;
  for (;;) {
    if (mask == 0) {
      if (b1 >= B) break;
      const int ml = m1 + lane * nrole;
      int b = b1, cnt = cnt1, base = base1;
      while (b < B && ml >= base + cnt) {
        base += cnt;
        if (++b < B) cnt = __ldg(miss_count + b);
      }
      bool valid = false;
      if (b < B)
        valid = miss_targets(L, miss_ids, miss_pos, victim, install, b, ml - base, k, P, sel_rows,
                             pool_rows, ctx_stride, ctx_len, my_from, my_to, my_to2, bad);
      mask = __ballot_sync(0xffffffffu, valid);
      // lane 31 holds the furthest index: the walk resumes from there
      b1 = __shfl_sync(0xffffffffu, b, 31);
      cnt1 = __shfl_sync(0xffffffffu, cnt, 31);
      base1 = __shfl_sync(0xffffffffu, base, 31);
      m1 += 32 * nrole;
      continue;
    }
    push_lanes(mask, my_from, my_to, my_to2, lane, pipe);
    mask = 0;
  }
}

// Every layer's misses handed out dynamically, layer after layer: a warp takes
// the next batch of kTicketRows misses (over all requests, concatenated) from the
// launch's ticket word, so warps that read host memory faster take more
// batches and every layer is done at about its share of the launch (measured
// on GB300 at 128 requests x 32,768 rows: with the misses dealt out evenly
// ahead of time, the fastest miss warps finished all four layers in half the
// time of the slowest, and a layer's completion waited for the slowest). The
// next ticket is fetched while the current batch is pushed. `prefix` holds the
// requests' exclusive miss-count prefix (B + 1 entries, shared memory).
__device__ __forceinline__ void gather_misses_dynamic(
    uint4* pool, const uint4* host, uint4* sel, int64_t pool_stride, int64_t host_stride,
    int64_t sel_stride, int layers, const int32_t* miss_ids, const int32_t* miss_pos,
    const int32_t* victim, const uint8_t* install, const int* prefix, int B, int k, int P,
    int sel_rows, int pool_rows, int64_t ctx_stride, const int32_t* ctx_len, uint32_t* ticket,
    int lane, RowPipe& pipe, int& bad) {
  const int total = prefix[B];
  const uint32_t nb = static_cast<uint32_t>((total + kTicketRows - 1) / kTicketRows);  // per layer
  const uint32_t end = nb * static_cast<uint32_t>(layers);
  uint32_t t = 0;
  if (lane == 0) t = atomicAdd(ticket, 1u);
  t = __shfl_sync(0xffffffffu, t, 0);
  int cur = 0;  // the layer this warp's rows belong to
  while (t < end) {
    uint32_t next = 0;
    if (lane == 0) next = atomicAdd(ticket, 1u);
    const int l = static_cast<int>(t / nb);
    for (; cur < l; ++cur) {  // every row of the earlier layers is pushed
      if (lane == 0) pipe.end_layer(cur);
      __syncwarp();
    }
    const GatherLayer L{pool + l * pool_stride, host + l * host_stride, sel + l * sel_stride};
    const int g = static_cast<int>(t % nb) * kTicketRows + lane;
    const uint4* from = nullptr;
    uint4* to = nullptr;
    uint4* to2 = nullptr;
    bool valid = false;
    int tag = kNoTag;
    if (lane < kTicketRows && g < total) {
      int lo = 0, hi = B;  // the request b with prefix[b] <= g < prefix[b + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= g) lo = mid;
        else hi = mid;
      }
      valid = miss_targets(L, miss_ids, miss_pos, victim, install, lo, g - prefix[lo], k, P,
                           sel_rows, pool_rows, ctx_stride, ctx_len, from, to, to2, bad);
      tag = l * B + lo;
      // a corrupt entry moves no row but still counts as arrived (its
      // request's attention then runs on, with the error reported)
      if (!valid && pipe.arrived) atomicAdd(pipe.arrived + tag, 1u);
    }
    push_lanes(__ballot_sync(0xffffffffu, valid), from, to, to2, lane, pipe, tag);
    t = __shfl_sync(0xffffffffu, next, 0);
  }
  for (; cur < layers - 1; ++cur) {  // the finish counts out of the last layer
    if (lane == 0) pipe.end_layer(cur);
    __syncwarp();
  }
}

// The positions: the pool row for a hit; for a miss, the host row only when
// the token repeats and this is not its first position (gather_misses serves
// first positions; requests without repeats, miss_rows == miss_count, skip
// misses outright). 32 positions at a time, one lookup per lane, pushed
// through the warp's pipe by lane 0.
__device__ __forceinline__ void gather_positions(
    const GatherLayer& L, const int32_t* src_map, const int32_t* miss_ids, const int32_t* miss_pos,
    const int32_t* miss_count, const int32_t* miss_rows, int B, int k, int P, int64_t ctx_stride,
    const int32_t* ctx_len, int w, int nrole, int lane, RowPipe& pipe, int& bad) {
  const int64_t rows = int64_t(B) * k;
  const int64_t step = int64_t(nrole) * 32;
  // the next batch's src_map entries are loaded before this batch's rows are
  // pushed, so the lookup does not stall the pipe
  int src_next = int64_t(w) * 32 + lane < rows ? __ldg(src_map + int64_t(w) * 32 + lane) : 0;
  for (int64_t r0 = int64_t(w) * 32; r0 < rows; r0 += step) {
    const int64_t r = r0 + lane;
    const int src = src_next;
    if (r + step < rows) src_next = __ldg(src_map + r + step);
    const uint4* from = nullptr;
    if (r < rows) {
      const int b = static_cast<int>(r / k);
      const int j = static_cast<int>(r - int64_t(b) * k);
      if (src >= 0) {
        if (src < P) from = L.pool + (int64_t(b) * P + src) * DSA_ROW_CHUNKS;
        else bad |= TS_DEVERR_SLOT_RANGE;
      } else if (src != INT_MIN) {
        const int M = __ldg(miss_count + b);
        const int t = -1 - src;
        const int64_t base = int64_t(b) * k;
        if (__ldg(miss_rows + b) != M && miss_first_pos(miss_ids + base, miss_pos + base, M, t) != j) {
          if (t < __ldg(ctx_len + b) && t < ctx_stride)
            from = L.host + (int64_t(b) * ctx_stride + t) * DSA_ROW_CHUNKS;
          else bad |= TS_DEVERR_ID_RANGE;
        }
      } else {
        bad |= TS_DEVERR_ID_RANGE;
      }
    }
    uint4* to = L.sel + r * DSA_ROW_CHUNKS;
    uint32_t mask = __ballot_sync(0xffffffffu, from != nullptr);
    while (mask) {
      const int q = __ffs(mask) - 1;
      mask &= mask - 1;
      const uint4* f = reinterpret_cast<const uint4*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(from), q));
      uint4* t = reinterpret_cast<uint4*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(to), q));
      if (lane == 0) pipe.push(f, t);
      __syncwarp();
    }
  }
}

// One launch for `layers` consecutive layers (layer l's pool, host rows and
// selection start l * pool_stride / host_stride / sel_stride pieces after
// layer 0's; a request's rows start sel_rows / pool_rows rows apart in the
// selection / pool: k and P, or P + k each for the staged layout, whose
// "selection" is the staging rows after the pool's slots), in two kinds of
// CTAs of kPipeWarps warps, every warp with its own RowPipe:
//   CTAs [0, miss_ctas): gather_misses, the host-link reads that set the
//     kernel's time (a few SMs keep the link busy);
//   the others: gather_positions, the pool hits (HBM), beside them.
// The two kinds write disjoint positions; with `victim` given the miss CTAs
// also install the code-1 misses into the pool (slots no hit of the step
// reads). Every warp finishes pushing a layer
// before it starts the next and keeps its pipe full across the boundary.
// With `done` given, each warp counts itself out of layer l in count[l] once
// its rows of the layer are written, and the last one resets the count and
// writes `seq` into done[l]: another stream's stream-memory wait on done[l]
// then orders the layer's consumers after its rows. The launch's own
// completion orders them for the per-layer call.
__global__ void __launch_bounds__(kGatherThreads, 1) gather_kernel(
    const int32_t* __restrict__ src_map, const int32_t* __restrict__ miss_ids,
    const int32_t* __restrict__ miss_pos, const int32_t* __restrict__ miss_count,
    const int32_t* __restrict__ miss_rows, const int32_t* __restrict__ victim,
    const uint8_t* __restrict__ install, int B, int k, uint4* pool, int P,
    const uint4* __restrict__ host, int64_t ctx_stride, const int32_t* __restrict__ ctx_len,
    uint4* __restrict__ sel, int layers, int64_t pool_stride, int64_t host_stride,
    int64_t sel_stride, uint32_t* __restrict__ done, uint32_t* __restrict__ count, uint32_t seq,
    int miss_ctas, int sel_rows, int pool_rows, uint32_t* ticket, uint32_t* arrived,
    int self_count, int32_t* err) {
  extern __shared__ __align__(128) uint8_t gather_smem[];
  __shared__ int scan_scratch[40];
  const int lane = threadIdx.x & 31;
  const int wc = threadIdx.x >> 5;  // warp in the CTA
  const int nw = static_cast<int>(gridDim.x) * kPipeWarps;
  const bool miss_cta = static_cast<int>(blockIdx.x) < miss_ctas;
  const int cta = miss_cta ? blockIdx.x : blockIdx.x - miss_ctas;
  const int w = cta * kPipeWarps + wc;
  const int nrole = (miss_cta ? miss_ctas : static_cast<int>(gridDim.x) - miss_ctas) * kPipeWarps;
  int bad = 0;
  if (arrived && threadIdx.x == 0) {
    // every CTA of the launch is running once the last one counts in: the
    // attention that waits for rows inside its kernel may start then
    uint32_t* started = arrived + size_t(layers) * B;
    if (atomicAdd(started, 1u) == gridDim.x - 1) atomicExch(started + 1, seq);
  }
  const bool counter = wc == kPipeWarps;  // the CTA's counting warp (no pipe)
  RowPipe pipe;
  if (lane == 0 && !counter)
    pipe.init(gather_smem + wc * kPipeWarpBytes, nw, count, done, seq, ticket, layers - 1,
              arrived, self_count != 0);
  __syncwarp();
  if (miss_cta && ticket) {
    // the requests' exclusive miss-count prefix, for the dynamic hand-out
    int* prefix = reinterpret_cast<int*>(gather_smem + kPipeSmemBytes);
    const int per = (B + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int b0 = min(static_cast<int>(threadIdx.x) * per, B), b1 = min(b0 + per, B);
    int c = 0;
    for (int b = b0; b < b1; ++b) c += min(max(__ldg(miss_count + b), 0), k);
    int total;
    int o = block_exclusive_scan(c, scan_scratch, &total);
    for (int b = b0; b < b1; ++b) {
      prefix[b] = o;
      o += min(max(__ldg(miss_count + b), 0), k);
    }
    if (threadIdx.x == 0) prefix[B] = total;
    __syncthreads();
    if (counter) {
      if (arrived && !self_count)
        count_arrivals(gather_smem, arrived, arrived + size_t(layers) * B + 2, lane);
    } else {
      gather_misses_dynamic(pool, host, sel, pool_stride, host_stride, sel_stride, layers,
                            miss_ids, miss_pos, victim, install, prefix, B, k, P, sel_rows,
                            pool_rows, ctx_stride, ctx_len, ticket, lane, pipe, bad);
      if (lane == 0) pipe.end_layer(layers - 1);
      __syncwarp();
    }
  }
  for (int l = 0; !counter && !(miss_cta && ticket) && l < layers; ++l) {
    const GatherLayer L{pool + l * pool_stride, host + l * host_stride, sel + l * sel_stride};
    if (miss_cta)
      gather_misses(L, miss_ids, miss_pos, miss_count, victim, install, B, k, P, sel_rows,
                    pool_rows, ctx_stride, ctx_len, w, nrole, lane, pipe, bad);
    else
      gather_positions(L, src_map, miss_ids, miss_pos, miss_count, miss_rows, B, k, P,
                       ctx_stride, ctx_len, w, nrole, lane, pipe, bad);
    if (lane == 0) pipe.end_layer(l);
    __syncwarp();
  }
  if (lane == 0 && !counter) {
    pipe.finish();
    if (pipe.failed) {
      bad |= TS_DEVERR_TIMEOUT;
      // the attention waiting for this launch's rows stops waiting
      if (arrived) atomicExch(arrived + size_t(layers) * B + 2, 1u);
    }
  }
  bad = __reduce_or_sync(0xffffffffu, bad);  // lookups are per lane
  if (bad && lane == 0) report(err, bad);
}

// The installs of every layer of the call, one CTA per request: its misses
// (the first miss_count[b] entries of its plan) 256 at a time with coalesced
// loads, then each warp copies the rows of its entries that need it, one
// after the other (72 pieces per row, lanes stride by 32). Layer l's
// selection and pool start sel_stride and pool_stride 16-byte pieces after
// layer l-1's. Requests hold a few hundred misses and the refill copies only
// the few whose victim slot the step read: scanning each request's own
// entries replaces a scan of all B x k positions (measured on GB300 at 128 x
// 32,768, the last layer's refill and metadata update: 35 us over all
// positions from one CTA per SM).
constexpr int kRefillThreads = 256;
__global__ void __launch_bounds__(kRefillThreads) refill_kernel(
    const int32_t* __restrict__ miss_ids, const int32_t* __restrict__ miss_pos,
    const int32_t* __restrict__ victim, const uint8_t* __restrict__ install,
    const int32_t* __restrict__ miss_count, int B, int k, const uint4* __restrict__ sel,
    uint4* __restrict__ pool, int P, int layers, int64_t sel_stride, int64_t pool_stride,
    int update_metadata, int32_t* __restrict__ pool_tags, int32_t* __restrict__ fifo_ptr,
    const int32_t* __restrict__ ptr_next, int S, int W, int min_install, int sel_rows,
    int pool_rows, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  const int M = min(max(__ldg(miss_count + b), 0), k);
  const int64_t base = int64_t(b) * k;
  for (int i0 = 0; i0 < M; i0 += kRefillThreads) {
    const int i = i0 + static_cast<int>(threadIdx.x);
    bool need = false;
    int64_t from_row = 0, to_row = 0;
    if (i < M) {
      const int code = __ldg(install + base + i);
      if (code) {
        const int v = __ldg(victim + base + i);
        const int j = __ldg(miss_pos + base + i);
        if (v < 0 || v >= P || j < 0 || j >= k) {
          report(err, TS_DEVERR_SLOT_RANGE);
        } else {
          if (update_metadata) pool_tags[int64_t(b) * P + v] = __ldg(miss_ids + base + i);
          // (rows with a lower code went in with the gather)
          need = code >= min_install;
          from_row = int64_t(b) * sel_rows + j;
          to_row = int64_t(b) * pool_rows + v;
        }
      }
    }
    uint32_t mask = __ballot_sync(0xffffffffu, need);
    while (mask) {
      const int q = __ffs(mask) - 1;
      mask &= mask - 1;
      const uint4* from = sel + __shfl_sync(0xffffffffu, from_row, q) * DSA_ROW_CHUNKS + lane;
      uint4* to = pool + __shfl_sync(0xffffffffu, to_row, q) * DSA_ROW_CHUNKS + lane;
      for (int l = 0; l < layers; ++l) {
        const uint4 x0 = ld_nc_v4(from);
        const uint4 x1 = ld_nc_v4(from + 32);
        st_v4(to, x0);
        st_v4(to + 32, x1);
        if (lane < DSA_ROW_CHUNKS - 64) st_v4(to + 64, ld_nc_v4(from + 64));
        from += sel_stride;
        to += pool_stride;
      }
    }
  }
  if (update_metadata) {
    for (int s = threadIdx.x; s < S; s += kRefillThreads) {
      const int p = __ldg(ptr_next + int64_t(b) * S + s);
      if (p < 0 || p >= W) {
        report(err, TS_DEVERR_PTR_RANGE);
        continue;
      }
      fifo_ptr[int64_t(b) * S + s] = p;
    }
  }
}


}  // namespace
}  // namespace dsakv

using namespace dsakv;

namespace dsakv {

ts_status gather_check(const int32_t* src_map, const int32_t* miss_ids, const int32_t* miss_pos,
                       const int32_t* miss_count, const int32_t* miss_rows, int B, int k,
                       const void* pool_l, int P, const void* host_l, int64_t ctx_stride,
                       const int32_t* ctx_len, void* sel_l) {
  if (!src_map || !miss_ids || !miss_pos || !miss_count || !miss_rows || !pool_l || !host_l ||
      !ctx_len || !sel_l)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || P <= 0 || ctx_stride <= 0) return TS_ERR_INVALID_ARG;
  if (!aligned16(pool_l) || !aligned16(host_l) || !aligned16(sel_l)) return TS_ERR_INVALID_ARG;
  return TS_OK;
}

// The launch's CTAs of the two kinds. The hit CTAs grow with the rows a layer
// moves (kHitCtas per kRowsPerHitUnit rows, at most kMaxUnits units). The miss
// CTAs: kMissCtas keep the host link busy while the host rows the launch reads
// span at most kWideHostBytes; over a wider span each zero-copy read waits
// longer (measured on GB300: random 1152-byte reads over 19 GB of page-locked
// memory from 8 SMs ran at 92 GB/s, from 24 at 126, where over 9.6 GB they ran
// at 124 and 207), so three units go to the misses, and never fewer units than
// the hits get. Measured per step: 4 x 4 x 1,048,576-row host KV (19 GB, 95 %
// misses) 0.81 ms with 8 + 16 CTAs, 0.47 with 24 + 16; 128 requests x 32,768
// rows (19 GB, 79 % hits) 4.44 ms with 8 + 16, 1.76 with 32 + 64.
struct GatherGrid {
  int miss, hit;  // multiples of kMissCtas and kHitCtas
};
const int64_t kRowsPerHitUnit = 65536;  // rows a layer moves per kHitCtas
const int kMaxUnits = 4;
const double kWideHostBytes = 12e9;  // host rows spanning more: 3 units of miss CTAs
GatherGrid gather_grid(int B, int k, double host_bytes) {
  const int64_t rows = int64_t(B) * k;
  const int h = static_cast<int>(
      std::min<int64_t>(kMaxUnits, std::max<int64_t>(1, (rows + kRowsPerHitUnit - 1) /
                                                            kRowsPerHitUnit)));
  const int m = std::max(h, host_bytes > kWideHostBytes ? 3 : 1);
  return {kMissCtas * m, kHitCtas * h};
}

ts_status gather_enqueue(const int32_t* src_map, const int32_t* miss_ids, const int32_t* miss_pos,
                         const int32_t* miss_count, const int32_t* miss_rows, int B, int k,
                         const void* pool_l, int P, const void* host_l, int64_t ctx_stride,
                         const int32_t* ctx_len, void* sel_l, int32_t* err, cudaStream_t stream,
                         int layers, size_t pool_layer_bytes, size_t host_layer_bytes,
                         size_t sel_layer_bytes, uint32_t* done, uint32_t* count, uint32_t seq,
                         const int32_t* victim, const uint8_t* install, bool staged,
                         uint32_t* ticket, uint32_t* arrived) {
  // At the decode_batch shape (32 x 2048 rows a layer, 9.7 GB of host KV):
  // kMissCtas + kHitCtas CTAs (24 SMs): the misses' share of them reads at
  // the host link's rate (measured alone: 8 SMs of bulk copies reach the
  // same ~205 GB/s as plain loads on 16-57 SMs), the rest copy the hits at
  // HBM speed, and each layer's attention fits in one wave on the SMs left
  // (decode_batch: 128 CTAs; with the gather on 57 SMs it took two).
  // Measured alternatives that did worse: plain loads on 3/8 of the SMs
  // (the earlier design, 0.549 vs 0.540 ms a step), other splits (9 + 15,
  // 10 + 14, 12 + 12, 6 + 18, 4 + 20 CTAs), 8 or 32 warps per CTA.
  // The staged layout moves only the misses (the attention reads the hits
  // from the pool itself): the miss CTAs alone, into the staging rows.
  // With `ticket` (the group step's), the misses are handed out dynamically
  // in layer order, which needs the requests' miss-count prefix in shared
  // memory beside the pipes.
  const bool dynamic = ticket && count && B <= kMaxDynamicB;
  // per-request arrival counts come from the dynamic hand-out's row tags
  if (arrived && !(dynamic && staged && gather_streams(B, layers))) return TS_ERR_INVALID_ARG;
  const size_t smem = kPipeSmemBytes + (dynamic ? (size_t(B) + 1) * 4 : 0);
  static std::atomic<uint64_t> smem_set{0};
  if (!raise_smem_limit(reinterpret_cast<const void*>(gather_kernel),
                        static_cast<int>(kPipeSmemBytes + (size_t(kMaxDynamicB) + 1) * 4),
                        smem_set))
    return TS_ERR_CUDA;
  const double host_bytes =
      double(host_layer_bytes ? host_layer_bytes : size_t(B) * size_t(ctx_stride) * DSA_ROW_BYTES) *
      layers;
  const GatherGrid grid = gather_grid(B, k, host_bytes);
  // Streamed arrival counts: with three or more units of miss CTAs the
  // launch keeps far more host rows in flight than the link needs, and the
  // pipe threads release their rows themselves (the counts then lag the rows
  // least); with fewer, every stall of a pipe costs link time, and the CTA's
  // counting warp releases them. Measured per step (GB300): 128 x 32,768
  // (32 miss CTAs) 1.55 ms with the pipes' own releases, 1.73 with counting
  // warps; 32 x 65,536 (8 miss CTAs) 0.73 and 0.55.
  const bool self_count = grid.miss >= 3 * kMissCtas;
  const int hit = staged ? 0 : grid.hit;
  const int pool_rows = staged ? P + k : P;
  const int sel_rows = staged ? P + k : k;
  uint4* pool = static_cast<uint4*>(const_cast<void*>(pool_l));
  uint4* sel = staged ? pool + size_t(P) * DSA_ROW_CHUNKS : static_cast<uint4*>(sel_l);
  if (staged) sel_layer_bytes = pool_layer_bytes;
  gather_kernel<<<grid.miss + hit, kGatherThreads, smem, stream>>>(
      src_map, miss_ids, miss_pos, miss_count, miss_rows, victim, install, B, k, pool, P,
      static_cast<const uint4*>(host_l), ctx_stride, ctx_len, sel, layers,
      int64_t(pool_layer_bytes / 16), int64_t(host_layer_bytes / 16),
      int64_t(sel_layer_bytes / 16), done, count, seq, grid.miss, sel_rows, pool_rows,
      dynamic ? ticket : nullptr, arrived, self_count ? 1 : 0, err);
  return launch_status();
}

ts_status stage_check(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* miss_count,
                      int B, int k, const void* pool_l, int P, const void* host_l,
                      int64_t ctx_stride, const int32_t* ctx_len) {
  if (!miss_ids || !miss_pos || !miss_count || !pool_l || !host_l || !ctx_len)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || P <= 0 || ctx_stride <= 0) return TS_ERR_INVALID_ARG;
  if (int64_t(B) * (int64_t(P) + k) >= (int64_t(1) << 31)) return TS_ERR_UNSUPPORTED;
  if (!aligned16(pool_l) || !aligned16(host_l)) return TS_ERR_INVALID_ARG;
  return TS_OK;
}

ts_status refill_check(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* victim,
                       const uint8_t* install, const int32_t* miss_count, int B, int k,
                       const void* sel_l, void* pool_l, int P, int update_metadata,
                       int32_t* pool_tags, int32_t* fifo_ptr, const int32_t* ptr_next, int S,
                       int W) {
  if (!miss_ids || !miss_pos || !victim || !install || !miss_count || !sel_l || !pool_l)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || P <= 0) return TS_ERR_INVALID_ARG;
  if (update_metadata && (!pool_tags || !fifo_ptr || !ptr_next || S <= 0 || W <= 0 || S * W != P))
    return TS_ERR_INVALID_ARG;
  if (!aligned16(sel_l) || !aligned16(pool_l)) return TS_ERR_INVALID_ARG;
  return TS_OK;
}

ts_status refill_enqueue(const int32_t* miss_ids, const int32_t* miss_pos, const int32_t* victim,
                         const uint8_t* install, const int32_t* miss_count, int B, int k,
                         const void* sel_l, void* pool_l, int P, int update_metadata,
                         int32_t* pool_tags, int32_t* fifo_ptr, const int32_t* ptr_next, int S,
                         int W, int32_t* err, cudaStream_t stream, int layers,
                         size_t sel_layer_bytes, size_t pool_layer_bytes, int min_install,
                         bool staged) {
  // one CTA per request (a small one: it fits beside an attention CTA). The
  // staged layout refills from the pool's own staging rows.
  const int pool_rows = staged ? P + k : P;
  const int sel_rows = staged ? P + k : k;
  const uint4* sel = staged ? static_cast<const uint4*>(pool_l) + size_t(P) * DSA_ROW_CHUNKS
                            : static_cast<const uint4*>(sel_l);
  if (staged) sel_layer_bytes = pool_layer_bytes;
  refill_kernel<<<static_cast<unsigned>(B), kRefillThreads, 0, stream>>>(
      miss_ids, miss_pos, victim, install, miss_count, B, k, sel, static_cast<uint4*>(pool_l), P,
      layers, int64_t(sel_layer_bytes / 16), int64_t(pool_layer_bytes / 16), update_metadata,
      pool_tags, fifo_ptr, ptr_next, S, W, min_install, sel_rows, pool_rows, err);
  return launch_status();
}

}  // namespace dsakv

extern "C" ts_status dsa_gather_kv(const int32_t* src_map, const int32_t* miss_ids,
                                   const int32_t* miss_pos, const int32_t* miss_count,
                                   const int32_t* miss_rows, int B, int k, const void* pool_l,
                                   int P, const void* host_l, int64_t ctx_stride,
                                   const int32_t* ctx_len, void* sel_l, int32_t* err,
                                   cudaStream_t stream) {
  const ts_status st = dsakv::gather_check(src_map, miss_ids, miss_pos, miss_count, miss_rows, B,
                                           k, pool_l, P, host_l, ctx_stride, ctx_len, sel_l);
  if (st != TS_OK) return st;
  return dsakv::gather_enqueue(src_map, miss_ids, miss_pos, miss_count, miss_rows, B, k, pool_l,
                               P, host_l, ctx_stride, ctx_len, sel_l, err, stream, 1, 0, 0, 0,
                               nullptr, nullptr, 0, nullptr, nullptr, false, nullptr, nullptr);
}

extern "C" ts_status dsa_stage_misses(const int32_t* miss_ids, const int32_t* miss_pos,
                                      const int32_t* miss_count, const int32_t* victim,
                                      const uint8_t* install, int B, int k, void* pool_l, int P,
                                      const void* host_l, int64_t ctx_stride,
                                      const int32_t* ctx_len, int32_t* err, cudaStream_t stream) {
  const ts_status st = dsakv::stage_check(miss_ids, miss_pos, miss_count, B, k, pool_l, P, host_l,
                                          ctx_stride, ctx_len);
  if (st != TS_OK) return st;
  if ((victim == nullptr) != (install == nullptr)) return TS_ERR_INVALID_ARG;
  return dsakv::gather_enqueue(nullptr, miss_ids, miss_pos, miss_count, nullptr, B, k, pool_l, P,
                               host_l, ctx_stride, ctx_len, nullptr, err, stream, 1, 0, 0, 0,
                               nullptr, nullptr, 0, victim, install, true, nullptr, nullptr);
}

extern "C" ts_status dsa_refill_pool(const int32_t* miss_ids, const int32_t* miss_pos,
                                     const int32_t* victim, const uint8_t* install,
                                     const int32_t* miss_count, int B, int k, const void* sel_l,
                                     void* pool_l, int P, int update_metadata, int32_t* pool_tags,
                                     int32_t* fifo_ptr, const int32_t* ptr_next, int S, int W,
                                     int32_t* err, cudaStream_t stream) {
  const ts_status st = dsakv::refill_check(miss_ids, miss_pos, victim, install, miss_count, B, k,
                                           sel_l, pool_l, P, update_metadata, pool_tags, fifo_ptr,
                                           ptr_next, S, W);
  if (st != TS_OK) return st;
  return dsakv::refill_enqueue(miss_ids, miss_pos, victim, install, miss_count, B, k, sel_l,
                               pool_l, P, update_metadata, pool_tags, fifo_ptr, ptr_next, S, W,
                               err, stream, 1, 0, 0, 1, false);
}

extern "C" ts_status dsa_refill_pool_staged(const int32_t* miss_ids, const int32_t* miss_pos,
                                            const int32_t* victim, const uint8_t* install,
                                            const int32_t* miss_count, int B, int k, void* pool_l,
                                            int P, int update_metadata, int32_t* pool_tags,
                                            int32_t* fifo_ptr, const int32_t* ptr_next, int S,
                                            int W, int32_t* err, cudaStream_t stream) {
  if (int64_t(B) * (int64_t(P) + k) >= (int64_t(1) << 31)) return TS_ERR_UNSUPPORTED;
  const ts_status st = dsakv::refill_check(miss_ids, miss_pos, victim, install, miss_count, B, k,
                                           pool_l, pool_l, P, update_metadata, pool_tags,
                                           fifo_ptr, ptr_next, S, W);
  if (st != TS_OK) return st;
  return dsakv::refill_enqueue(miss_ids, miss_pos, victim, install, miss_count, B, k, nullptr,
                               pool_l, P, update_metadata, pool_tags, fifo_ptr, ptr_next, S, W,
                               err, stream, 1, 0, 0, 1, true);
}

// ---------------------------------------------------------------------------
// ts_copy: a byte copy done by the SMs (16-byte loads and stores), between any
// two device-accessible buffers: device memory or registered host memory.
// ---------------------------------------------------------------------------
namespace dsakv {
namespace {

__global__ void __launch_bounds__(512) sm_copy_kernel(const uint4* __restrict__ src,
                                                      uint4* __restrict__ dst, int64_t n16) {
  const int64_t step = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += step * 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * step < n16) v[u] = ld_nc_v4(src + i + u * step);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * step < n16) st_v4(dst + i + u * step, v[u]);
  }
}

}  // namespace
}  // namespace dsakv

extern "C" ts_status ts_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (!dst || !src) return TS_ERR_INVALID_ARG;
  if (!aligned16(dst) || !aligned16(src) || (bytes & 15u) != 0) return TS_ERR_INVALID_ARG;
  if (bytes == 0) return TS_OK;
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  int64_t blocks = (n16 + 4 * 512 - 1) / (4 * 512);
  const int64_t cap = int64_t(sm_count()) * 2;
  if (blocks > cap) blocks = cap;
  sm_copy_kernel<<<static_cast<unsigned>(blocks), 512, 0, stream>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return launch_status();
}
