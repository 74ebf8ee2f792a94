// ts_topk: the k positions of largest Lightning-Indexer score per request
// (GLM-5.2 shared-Indexer KV Cache Offload, §2.1: the indexer selects the 2048
// history positions most relevant to the query, and sparse attention reads
// only those). Ties go to the lower position; output in ascending position.
//
// Radix select on the order-preserving 32-bit key of every score:
//   hist   : histogram of the top 12 bits of the key;
//   select : find the threshold bin (the bin holding the k-th largest key),
//            mark the positions of higher bins in a bitmap (one 32-bit word per
//            32 positions, built by a warp ballot) and list the threshold
//            bin's (key, position) pairs as candidates;
//   finish : resolve the threshold inside the candidate list (two more 10-bit
//            digits, then the lowest positions among exact ties), set their
//            bits, and write the set positions of the bitmap in order: the
//            output comes out sorted without a sort.
// Contexts up to 262,144 positions: one launch, one thread-block cluster of
// 1 to 8 CTAs per request, each holding the keys of up to 32,768 positions in shared
// memory; the CTAs merge their histograms through distributed shared memory,
// rank 0 resolves the exact threshold and broadcasts it, and every CTA writes
// its own slice of the sorted output. Longer contexts: hist and select spread
// over many CTAs per request (8,192 positions each); the last select CTA of a
// request to finish (a completion counter) resolves the threshold and each
// chunk's first output slot, and an output launch writes every chunk's
// positions in order, one CTA per chunk.
#include <mutex>

#include "common.cuh"
#include "ops.h"

namespace dsakv {
namespace {

constexpr int kBins = 4096;    // top 12 bits of the key
constexpr int kChunk = 8192;   // positions per CTA in the multi-CTA select
constexpr int kSlice = 32768;  // positions per CTA of the cluster kernel (at most)
constexpr int kClusterMaxG = 8;   // CTAs per request's cluster (the portable cluster size)
constexpr int kClusterFillG = 4;  // at most this many only to fill the SMs (short contexts)
constexpr int kHistChunk = 32768;  // positions per CTA in the multi-CTA hist (one wave at 4 x 1M)
constexpr int kThreads = 512;  // multi-CTA kernels
constexpr int kMaxK = 8192;
constexpr int kFinishCandCap = 4096;  // ... by the multi-CTA finish
constexpr uint32_t kAll = 0xFFFFFFFFu;

struct TopkWs {
  uint32_t* hist;        // [B][kBins]
  uint32_t* cand_count;  // [B] candidates listed, then [B] select CTAs done
  uint64_t* cand;        // [B][max_ctx]  (key << 32 | position)
  uint32_t* bitmap;      // [B][words]
  uint32_t* chunk;       // [B][chunks] selected positions of each select chunk, then its offset
  int64_t words, chunks;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline TopkWs carve(void* ws, int B, int max_ctx) {
  TopkWs w;
  char* p = static_cast<char*>(ws);
  w.hist = reinterpret_cast<uint32_t*>(p);
  p += align256(size_t(B) * kBins * 4);
  w.cand_count = reinterpret_cast<uint32_t*>(p);
  p += align256(size_t(B) * 8);
  w.cand = reinterpret_cast<uint64_t*>(p);
  p += align256(size_t(B) * max_ctx * 8);
  w.bitmap = reinterpret_cast<uint32_t*>(p);
  w.words = (max_ctx + 31) / 32;
  p += align256(size_t(B) * w.words * 4);
  w.chunk = reinterpret_cast<uint32_t*>(p);
  w.chunks = (max_ctx + kChunk - 1) / kChunk;
  return w;
}

inline size_t counters_bytes(int B) {
  return align256(size_t(B) * kBins * 4) + align256(size_t(B) * 8);
}

// Order-preserving key: a larger float gives a larger unsigned key. -0.0 is
// +0.0; NaN gets key 0 (ranks lowest) and is reported.
__device__ __forceinline__ uint32_t score_key(float f, bool& nan) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) {
    nan = true;
    return 0u;
  }
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool ctx_ok(int n, int k, int max_ctx) { return n >= k && n <= max_ctx; }

// The bin t of an nbins histogram (walked from the preferred end: high bins
// first when high_first) with before(t) < need <= before(t) + hist[t]; also
// returns before(t) and hist[t]. Block-wide; every thread gets the result.
// sbuf holds >= 44 ints.
__device__ void select_bin(const uint32_t* hist, int nbins, bool high_first, int need, int* sbuf,
                           int* bin_out, int* before_out, int* count_out) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  int tot = 0;
  for (int j = 0; j < per; ++j) {
    const int r = threadIdx.x * per + j;  // rank in preference order
    if (r < nbins) tot += static_cast<int>(hist[high_first ? nbins - 1 - r : r]);
  }
  int total;
  const int ex = block_exclusive_scan(tot, sbuf, &total);
  if (threadIdx.x == 0) {
    sbuf[40] = -1;
    sbuf[41] = 0;
    sbuf[42] = 0;
  }
  __syncthreads();
  int cum = ex;
  for (int j = 0; j < per; ++j) {
    const int r = threadIdx.x * per + j;
    if (r >= nbins) break;
    const int bin = high_first ? nbins - 1 - r : r;
    const int h = static_cast<int>(hist[bin]);
    if (cum < need && cum + h >= need) {
      sbuf[40] = bin;
      sbuf[41] = cum;
      sbuf[42] = h;
    }
    cum += h;
  }
  __syncthreads();
  *bin_out = sbuf[40];
  *before_out = sbuf[41];
  *count_out = sbuf[42];
  __syncthreads();
}

// Candidate lists: the first `cap` entries in shared memory, the rest in the
// global workspace (cap = 0: all global).
struct Cands {
  const uint64_t* smem;
  const uint64_t* glob;
  uint32_t cap;
  __device__ __forceinline__ uint64_t operator()(uint32_t i) const {
    return i < cap ? smem[i] : __ldcg(glob + i);
  }
};

// A candidate list in up to four global segments (one per CTA of a cluster):
// entry i lies in the segment s with off[s] <= i < off[s+1].
struct SegCands {
  const uint64_t* seg[kClusterMaxG];
  uint32_t off[kClusterMaxG + 1];
  __device__ __forceinline__ uint64_t operator()(uint32_t i) const {
    int s = 0;
#pragma unroll
    for (int g = 1; g < kClusterMaxG; ++g) s += i >= off[g];
    return __ldcg(seg[s] + (i - off[s]));
  }
};

// Histogram of a digit of the candidates satisfying pred, then select_bin.
template <typename C, typename Pred, typename Digit>
__device__ void cand_digit(const C& cand, uint32_t c, int nbins, bool high_first, int need,
                           Pred pred, Digit digit, uint32_t* hist, int* sbuf, int* t_out,
                           int* before_out, int* count_out) {
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
    const uint64_t e = cand(i);
    if (pred(e)) atomicAdd(&hist[digit(e)], 1u);
  }
  __syncthreads();
  select_bin(hist, nbins, high_first, need, sbuf, t_out, before_out, count_out);
}

// The exact threshold inside a request's candidate list (all candidates share
// the 12-bit bin t1; need1 of them are taken): a candidate is taken when its
// key > *T, or key == *T and position <= *cut. Block-wide; hist: >= 2048
// words of shared memory.
template <typename C>
__device__ void resolve_threshold(const C& cand, uint32_t c, int t1, int need1, uint32_t* hist,
                                  int* sbuf, uint32_t* T_out, uint32_t* cut_out) {
  uint32_t T = 0, cut = kAll;  // need1 >= c: every candidate
  if (need1 < static_cast<int>(c)) {
    int t2, before2, cnt2, t3, before3, cnt3;
    cand_digit(
        cand, c, 1024, true, need1, [](uint64_t) { return true; },
        [](uint64_t e) { return static_cast<int>((e >> 42) & 1023u); }, hist, sbuf, &t2, &before2,
        &cnt2);
    const int need2 = need1 - before2;
    cand_digit(
        cand, c, 1024, true, need2,
        [t2](uint64_t e) { return static_cast<int>((e >> 42) & 1023u) == t2; },
        [](uint64_t e) { return static_cast<int>((e >> 32) & 1023u); }, hist, sbuf, &t3,
        &before3, &cnt3);
    const int need3 = need2 - before3;  // exact ties to take
    T = (static_cast<uint32_t>(t1) << 20) | (static_cast<uint32_t>(t2) << 10) |
        static_cast<uint32_t>(t3);
    if (need3 < cnt3) {
      // the lowest positions among the exact ties: three digits of the position
      auto is_tie = [T](uint64_t e) { return static_cast<uint32_t>(e >> 32) == T; };
      int pa, ba, ca, pb, bb, cb, pc, bc, cc;
      cand_digit(
          cand, c, 2048, false, need3, is_tie,
          [](uint64_t e) { return static_cast<int>((static_cast<uint32_t>(e) >> 20) & 2047u); },
          hist, sbuf, &pa, &ba, &ca);
      cand_digit(
          cand, c, 1024, false, need3 - ba,
          [is_tie, pa](uint64_t e) {
            return is_tie(e) && static_cast<int>((static_cast<uint32_t>(e) >> 20) & 2047u) == pa;
          },
          [](uint64_t e) { return static_cast<int>((static_cast<uint32_t>(e) >> 10) & 1023u); },
          hist, sbuf, &pb, &bb, &cb);
      cand_digit(
          cand, c, 1024, false, need3 - ba - bb,
          [is_tie, pa, pb](uint64_t e) {
            const uint32_t p = static_cast<uint32_t>(e);
            return is_tie(e) && static_cast<int>((p >> 20) & 2047u) == pa &&
                   static_cast<int>((p >> 10) & 1023u) == pb;
          },
          [](uint64_t e) { return static_cast<int>(static_cast<uint32_t>(e) & 1023u); }, hist,
          sbuf, &pc, &bc, &cc);
      cut = (static_cast<uint32_t>(pa) << 20) | (static_cast<uint32_t>(pb) << 10) |
            static_cast<uint32_t>(pc);
    }
  }
  *T_out = T;
  *cut_out = cut;
}

__device__ __forceinline__ bool taken(uint64_t e, uint32_t T, uint32_t cut) {
  const uint32_t key = static_cast<uint32_t>(e >> 32), pos = static_cast<uint32_t>(e);
  return key > T || (key == T && pos <= cut);
}

// Resolve the threshold, set the chosen candidates' bits in the request's
// global bitmap and add them to their chunks' counts (which hold each select
// chunk's positions above the threshold bin), then turn the counts into each
// chunk's first output slot (an exclusive scan over the request's chunks).
// topk_output_kernel then writes every chunk's positions in order, one CTA
// per chunk. A total other than k sets TS_DEVERR_COUNT, writes -1 ids and
// marks every chunk so that nothing more is written.
template <typename C>
__device__ void finish_chunks(const C& cand, uint32_t c, int t1, int need1, uint32_t* bits,
                              uint32_t* counts, int n, int k, int32_t* out, uint32_t* hist,
                              int* sbuf, int32_t* err) {
  uint32_t T, cut;
  resolve_threshold(cand, c, t1, need1, hist, sbuf, &T, &cut);
  for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
    const uint64_t e = cand(i);
    if (taken(e, T, cut)) {
      const uint32_t pos = static_cast<uint32_t>(e);
      atomicOr(bits + (pos >> 5), 1u << (pos & 31));
      atomicAdd(counts + pos / kChunk, 1u);
    }
  }
  __syncthreads();
  const int nch = (n + kChunk - 1) / kChunk;
  const int per = (nch + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int j0 = min(static_cast<int>(threadIdx.x) * per, nch), j1 = min(j0 + per, nch);
  int cnt = 0;
  for (int j = j0; j < j1; ++j) cnt += static_cast<int>(__ldcg(counts + j));
  int total;
  int off = block_exclusive_scan(cnt, sbuf, &total);
  if (total != k) {
    if (threadIdx.x == 0) report(err, TS_DEVERR_COUNT);
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    for (int j = threadIdx.x; j < nch; j += blockDim.x) counts[j] = kAll;
    return;
  }
  for (int j = j0; j < j1; ++j) {
    const int c_j = static_cast<int>(__ldcg(counts + j));
    counts[j] = static_cast<uint32_t>(off);
    off += c_j;
  }
}

// ---------------------------------------------------------------------------
// contexts up to kClusterMaxCtx: one cluster of G = ceil(ctx / 32768) CTAs
// per request, every CTA holding the keys of its 32,768-position slice in
// shared memory; histograms merge through distributed shared memory.
// ---------------------------------------------------------------------------
constexpr int kClusterMaxCtx = kSlice * kClusterMaxG;
constexpr int kClThreads = 1024;
constexpr int kClCandCap = 4096;  // candidates kept in shared memory by rank 0

struct ClSmem {
  uint32_t keys[kSlice];         // this CTA's keys
  uint32_t hist[kBins];          // this CTA's histogram (read by the cluster)
  uint32_t tot[kBins];           // the merged histogram, then digit histograms
  uint32_t bits[kSlice / 32];    // this CTA's part of the bitmap
  uint64_t cand[kClCandCap];     // rank 0: the request's candidates
  int sbuf[64];
  uint32_t ncand;                // candidates of this CTA (in the global list)
  uint32_t nsel;                 // positions this CTA selected
  uint32_t thr[2];               // (T, cut), broadcast by rank 0
};

__global__ void __launch_bounds__(kClThreads, 1) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t ctx_stride, const int32_t* __restrict__ ctx_len,
    int k, int max_ctx, int slice, TopkWs ws, int32_t* __restrict__ ids, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ClSmem& sm = *reinterpret_cast<ClSmem*>(smem_raw);
  const int G = gridDim.x;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  const bool ok = ctx_ok(n, k, max_ctx);  // uniform over the cluster
  int32_t* out = ids + int64_t(b) * k;
  const int lo = static_cast<int>(rank) * slice;  // slice <= kSlice
  const int hi = ok ? min(lo + slice, n) : lo;
  const int len = max(hi - lo, 0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t* gcand = ws.cand + int64_t(b) * max_ctx + lo;  // this CTA's global candidate list

  for (int i = tid; i < kBins; i += kClThreads) sm.hist[i] = 0;
  if (tid == 0) {
    sm.ncand = 0;
    sm.nsel = 0;
  }
  __syncthreads();
  // keys and histogram of the slice (8 loads in flight per thread)
  bool nan = false;
  const float* row = scores + int64_t(b) * ctx_stride + lo;
  for (int base = warp * 256; base < len; base += (kClThreads / 32) * 256) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * 32 + lane;
      v[u] = i < len ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * 32 + lane;
      if (i < len) {
        const uint32_t key = score_key(v[u], nan);
        sm.keys[i] = key;
        atomicAdd(&sm.hist[key >> 20], 1u);
      }
    }
  }
  if (nan) report(err, TS_DEVERR_NAN);
  cluster_sync_all();

  // merged histogram: every CTA sums the cluster's histograms
  for (int i4 = tid; i4 < kBins / 4; i4 += kClThreads) {
    uint4 acc = make_uint4(0, 0, 0, 0);
    for (int g = 0; g < G; ++g) {
      const uint4 h = ld_dsmem_u4(dsmem_addr(&sm.hist[4 * i4], g));
      acc.x += h.x;
      acc.y += h.y;
      acc.z += h.z;
      acc.w += h.w;
    }
    *reinterpret_cast<uint4*>(&sm.tot[4 * i4]) = acc;
  }
  __syncthreads();
  int t1 = 0, above = 0, cnt1 = 0;
  if (ok) select_bin(sm.tot, kBins, true, k, sm.sbuf, &t1, &above, &cnt1);
  else __syncthreads();

  // bitmap words above the threshold bin; the bin's candidates to the global list
  for (int base = warp * 128; base < len; base += (kClThreads / 32) * 128) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * 32 + lane;
      const uint32_t key = i < len ? sm.keys[i] : 0u;
      const int bin = i < len ? static_cast<int>(key >> 20) : -1;
      const uint32_t above_mask = __ballot_sync(0xffffffffu, bin > t1);
      const uint32_t tie_mask = __ballot_sync(0xffffffffu, bin == t1);
      if (lane == 0 && base + u * 32 < len) sm.bits[(base + u * 32) >> 5] = above_mask;
      if (tie_mask) {
        uint32_t pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(&sm.ncand, __popc(tie_mask));
        pos0 = __shfl_sync(0xffffffffu, pos0, 0);
        if (bin == t1)
          gcand[pos0 + __popc(tie_mask & ((1u << lane) - 1u))] =
              (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(lo + i);
      }
    }
  }
  cluster_sync_all();  // candidate lists and their counts are visible to rank 0

  if (rank == 0 && ok) {
    SegCands cl;
    cl.off[0] = 0;
    for (int g = 0; g < kClusterMaxG; ++g) {
      const uint32_t cg = g < G ? ld_dsmem_u32(dsmem_addr(&sm.ncand, g)) : 0u;
      cl.seg[g] = ws.cand + int64_t(b) * max_ctx + int64_t(g) * slice;
      cl.off[g + 1] = cl.off[g] + cg;
    }
    const uint32_t c = cl.off[kClusterMaxG];
    uint32_t T, cut;
    if (c <= kClCandCap) {
      // the common case: the whole list in shared memory
      for (uint32_t i = tid; i < c; i += kClThreads) sm.cand[i] = cl(i);
      __syncthreads();
      Cands cs{sm.cand, nullptr, kClCandCap};
      resolve_threshold(cs, c, t1, k - above, sm.tot, sm.sbuf, &T, &cut);
    } else {
      resolve_threshold(cl, c, t1, k - above, sm.tot, sm.sbuf, &T, &cut);
    }
    if (tid < G) {
      st_dsmem_u32(dsmem_addr(&sm.thr[0], tid), T);
      st_dsmem_u32(dsmem_addr(&sm.thr[1], tid), cut);
    }
  }
  cluster_sync_all();  // (T, cut) everywhere

  // every CTA sets its own candidates' bits and counts its selected positions
  if (ok) {
    const uint32_t T = sm.thr[0], cut = sm.thr[1];
    for (uint32_t i = tid; i < sm.ncand; i += kClThreads) {
      const uint64_t e = __ldcg(gcand + i);
      if (taken(e, T, cut)) {
        const uint32_t p = static_cast<uint32_t>(e) - lo;
        atomicOr(&sm.bits[p >> 5], 1u << (p & 31));
      }
    }
  }
  __syncthreads();
  const int nwords = (len + 31) / 32;
  const int per = (nwords + kClThreads - 1) / kClThreads;
  const int w0 = tid * per, w1 = min(w0 + per, nwords);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(sm.bits[w]);
  int total;
  int pos = block_exclusive_scan(cnt, sm.sbuf, &total);
  if (tid == 0) sm.nsel = total;
  cluster_sync_all();  // every CTA's count is visible

  int offset = 0, all = 0;
  for (int g = 0; g < G; ++g) {
    const int cg = static_cast<int>(ld_dsmem_u32(dsmem_addr(&sm.nsel, g)));
    if (g < static_cast<int>(rank)) offset += cg;
    all += cg;
  }
  if (!ok || all != k) {
    if (rank == 0) {
      for (int i = tid; i < k; i += kClThreads) out[i] = -1;
      if (tid == 0) report(err, ok ? TS_DEVERR_COUNT : TS_DEVERR_CTX);
    }
  } else {
    pos += offset;
    for (int w = w0; w < w1; ++w) {
      uint32_t m = sm.bits[w];
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1;
        out[pos++] = lo + w * 32 + bit;
      }
    }
  }
  cluster_sync_all();  // no CTA leaves while others may read its shared memory
}

// ---------------------------------------------------------------------------
// many CTAs per request
// ---------------------------------------------------------------------------
// Scores cluster in few bins, so shared-memory atomics on one histogram
// collide; every pair of warps counts into its own copy (8 copies, 128 KB of
// dynamic shared memory) and the copies are summed when flushed.
constexpr int kHistCopies = kThreads / 64;

__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const float* __restrict__ scores,
                                                             int64_t ctx_stride,
                                                             const int32_t* __restrict__ ctx_len,
                                                             int k, int max_ctx, TopkWs ws,
                                                             int32_t* err) {
  extern __shared__ __align__(16) uint32_t hcopies[];  // [kHistCopies][kBins]
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  if (!ctx_ok(n, k, max_ctx)) return;
  const int64_t start = int64_t(blockIdx.x) * kHistChunk;
  if (start >= n) return;
  const int64_t end = min(start + int64_t(kHistChunk), int64_t(n));
  for (int i = threadIdx.x; i < kHistCopies * kBins; i += kThreads) hcopies[i] = 0;
  __syncthreads();
  const float* row = scores + int64_t(b) * ctx_stride;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* h = hcopies + (warp >> 1) * kBins;
  bool nan = false;
  for (int64_t base = start + warp * 256; base < end; base += (kThreads / 32) * 256) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = base + u * 32 + lane;
      v[u] = i < end ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = base + u * 32 + lane;
      if (i < end) atomicAdd(&h[score_key(v[u], nan) >> 20], 1u);
    }
  }
  if (nan) report(err, TS_DEVERR_NAN);
  __syncthreads();
  uint32_t* gh = ws.hist + int64_t(b) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads) {
    uint32_t sum = 0;
#pragma unroll
    for (int cpy = 0; cpy < kHistCopies; ++cpy) sum += hcopies[cpy * kBins + i];
    if (sum) atomicAdd(&gh[i], sum);
  }
}

__global__ void __launch_bounds__(kThreads) topk_select_kernel(
    const float* __restrict__ scores, int64_t ctx_stride, const int32_t* __restrict__ ctx_len,
    int k, int max_ctx, TopkWs ws, int32_t* __restrict__ ids, int32_t* err) {
  __shared__ int sbuf[64];
  __shared__ uint32_t dig[2048];
  __shared__ uint64_t cand_s[kFinishCandCap];
  __shared__ int last;
  __shared__ uint32_t chunk_above;
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  if (!ctx_ok(n, k, max_ctx)) {
    if (blockIdx.x == 0) {
      int32_t* out = ids + int64_t(b) * k;
      for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
      if (threadIdx.x == 0) report(err, TS_DEVERR_CTX);
    }
    return;
  }
  const int64_t start = int64_t(blockIdx.x) * kChunk;
  if (start >= n) return;
  if (threadIdx.x == 0) chunk_above = 0;  // (select_bin's barriers come before its use)
  // threshold bin from the request's histogram
  int t1, above, cnt1;
  select_bin(ws.hist + int64_t(b) * kBins, kBins, true, k, sbuf, &t1, &above, &cnt1);
  const int64_t end = min(start + int64_t(kChunk), int64_t(n));
  const float* row = scores + int64_t(b) * ctx_stride;
  uint32_t* bits = ws.bitmap + int64_t(b) * ws.words;
  uint64_t* cand = ws.cand + int64_t(b) * max_ctx;
  const int lane = threadIdx.x & 31;
  // each warp covers 4 x 32 consecutive positions per iteration: 4 bitmap words
  const int warp = threadIdx.x >> 5;
  uint32_t n_above = 0;  // this warp's positions above the threshold bin
  for (int64_t base = start + warp * 128; base < end; base += (kThreads / 32) * 128) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = base + u * 32 + lane;
      v[u] = i < end ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = base + u * 32 + lane;
      bool nan = false;
      uint32_t key = 0;
      int bin = -1;
      if (i < end) {
        key = score_key(v[u], nan);
        bin = static_cast<int>(key >> 20);
      }
      const uint32_t above_mask = __ballot_sync(0xffffffffu, bin > t1);
      const uint32_t tie_mask = __ballot_sync(0xffffffffu, bin == t1);
      n_above += __popc(above_mask);
      if (lane == 0 && base + u * 32 < end) bits[(base + u * 32) >> 5] = above_mask;
      if (tie_mask) {
        uint32_t pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(ws.cand_count + b, __popc(tie_mask));
        pos0 = __shfl_sync(0xffffffffu, pos0, 0);
        if (bin == t1) {
          const uint32_t off = __popc(tie_mask & ((1u << lane) - 1u));
          cand[pos0 + off] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
        }
      }
    }
  }
  // the chunk's count of positions above the bin, then the last CTA of this
  // request to get here runs the finish
  if (lane == 0) atomicAdd(&chunk_above, n_above);
  __syncthreads();
  if (threadIdx.x == 0) ws.chunk[int64_t(b) * ws.chunks + blockIdx.x] = chunk_above;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t chunks = static_cast<uint32_t>((int64_t(n) + kChunk - 1) / kChunk);
    last = atomicAdd(ws.cand_count + gridDim.y + b, 1u) == chunks - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const uint32_t c = __ldcg(ws.cand_count + b);
  // the finish reads the candidate list several times: keep its head in
  // shared memory
  for (uint32_t i = threadIdx.x; i < c && i < kFinishCandCap; i += blockDim.x)
    cand_s[i] = __ldcg(cand + i);
  __syncthreads();
  Cands cl{cand_s, cand, kFinishCandCap};
  finish_chunks(cl, c, t1, k - above, bits, ws.chunk + int64_t(b) * ws.chunks, n, k,
                ids + int64_t(b) * k, dig, sbuf, err);
}

// Each select chunk's selected positions, in order, at the chunk's first
// output slot (finish_chunks): one CTA per chunk, one bitmap word per thread.
constexpr int kOutThreads = kChunk / 32;
__global__ void __launch_bounds__(kOutThreads) topk_output_kernel(
    const int32_t* __restrict__ ctx_len, int k, int max_ctx, TopkWs ws,
    int32_t* __restrict__ ids) {
  __shared__ int scratch[40];
  const int b = blockIdx.y, j = blockIdx.x;
  const int n = ctx_len[b];
  if (!ctx_ok(n, k, max_ctx)) return;  // (the select kernel wrote the request's -1 ids)
  const int64_t start = int64_t(j) * kChunk;
  if (start >= n) return;
  const uint32_t off = __ldcg(ws.chunk + int64_t(b) * ws.chunks + j);
  if (off == kAll) return;  // (a count other than k: reported, ids -1)
  const int64_t nwords = (int64_t(n) + 31) / 32;
  const int64_t w = start / 32 + threadIdx.x;
  uint32_t m = w < nwords ? __ldcg(ws.bitmap + int64_t(b) * ws.words + w) : 0u;
  int total;
  const int pos = block_exclusive_scan(__popc(m), scratch, &total);
  int32_t* o = ids + int64_t(b) * k + off + pos;
  while (m) {
    const int bit = __ffs(m) - 1;
    m &= m - 1;
    *o++ = static_cast<int32_t>(w * 32 + bit);
  }
}


// Launch the top-k on a workspace laid out by carve().
ts_status launch_topk(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                      int max_ctx, int k, int32_t* ids, void* ws, int32_t* err,
                      cudaStream_t stream) {
  TopkWs w = carve(ws, B, max_ctx);
  if (max_ctx <= kClusterMaxCtx) {
    static std::atomic<uint64_t> smem_set{0};
    if (!raise_smem_limit(reinterpret_cast<const void*>(topk_cluster_kernel),
                          int(sizeof(ClSmem)), smem_set))
      return TS_ERR_CUDA;
    // enough CTAs per request for slices of at most kSlice positions (a
    // multiple of 1024), and, when the requests are few, to fill half of the
    // SMs (up to kClusterFillG; the other half stays free for the kernels of
    // the previous step still running, which would otherwise delay this
    // launch)
    int G = (max_ctx + kSlice - 1) / kSlice;
    const int fill = sm_count() / (2 * B);
    if (fill > G) G = max(G, min(fill, kClusterFillG));
    const int slice = ((max_ctx + G - 1) / G + 1023) / 1024 * 1024;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, B, 1);
    cfg.blockDim = dim3(kClThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(ClSmem);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = G;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // clusters above kClusterFillG CTAs of this size need a GPC with that many
    // free SMs: asked of the device once per size (contexts that need them
    // otherwise take the multi-launch path below)
    bool fits = true;
    if (G > kClusterFillG) {
      static std::atomic<int> fit_known[kClusterMaxG + 1];  // 0 unknown, 1 yes, 2 no
      int known = fit_known[G].load(std::memory_order_relaxed);
      if (known == 0) {
        int n = 0;
        known = cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel, &cfg) == cudaSuccess &&
                        n > 0
                    ? 1
                    : 2;
        cudaGetLastError();
        fit_known[G].store(known, std::memory_order_relaxed);
      }
      fits = known == 1;
    }
    if (fits) {
      if (cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, ctx_stride, ctx_len, k, max_ctx,
                             slice, w, ids, err) != cudaSuccess)
        return TS_ERR_CUDA;
      return TS_OK;
    }
  }
  // histograms, list counters and completion counters start at zero
  if (cudaMemsetAsync(ws, 0, counters_bytes(B), stream) != cudaSuccess) return TS_ERR_CUDA;
  const dim3 grid((max_ctx + kChunk - 1) / kChunk, B);
  static std::atomic<uint64_t> hist_smem_set{0};
  if (!raise_smem_limit(reinterpret_cast<const void*>(topk_hist_kernel), kHistCopies * kBins * 4,
                        hist_smem_set))
    return TS_ERR_CUDA;
  const dim3 hgrid((max_ctx + kHistChunk - 1) / kHistChunk, B);
  topk_hist_kernel<<<hgrid, kThreads, kHistCopies * kBins * 4, stream>>>(scores, ctx_stride,
                                                                         ctx_len, k, max_ctx, w,
                                                                         err);
  topk_select_kernel<<<grid, kThreads, 0, stream>>>(scores, ctx_stride, ctx_len, k, max_ctx, w,
                                                    ids, err);
  topk_output_kernel<<<grid, kOutThreads, 0, stream>>>(ctx_len, k, max_ctx, w, ids);
  return launch_status();
}

ts_status check_topk_args(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                          int max_ctx, int k, int32_t* ids) {
  if (!scores || !ctx_len || !ids) return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || max_ctx < k || ctx_stride < max_ctx) return TS_ERR_INVALID_ARG;
  if (k > kMaxK || B > 65535) return TS_ERR_UNSUPPORTED;
  if (!aligned16(scores) || (ctx_stride & 3) != 0) return TS_ERR_INVALID_ARG;
  return TS_OK;
}

}  // namespace
}  // namespace dsakv

using namespace dsakv;

extern "C" size_t ts_topk_workspace_size(int B, int max_ctx, int k) {
  (void)k;
  if (B <= 0 || max_ctx <= 0) return 0;
  const int64_t words = (int64_t(max_ctx) + 31) / 32;
  const int64_t chunks = (int64_t(max_ctx) + kChunk - 1) / kChunk;
  return align256(size_t(B) * kBins * 4) + align256(size_t(B) * 8) +
         align256(size_t(B) * max_ctx * 8) + align256(size_t(B) * words * 4) +
         align256(size_t(B) * chunks * 4);
}

namespace dsakv {

ts_status topk_check(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                     int max_ctx, int k, int32_t* ids, const void* ws, size_t ws_bytes) {
  const ts_status st = check_topk_args(scores, ctx_stride, ctx_len, B, max_ctx, k, ids);
  if (st != TS_OK) return st;
  if (!ws) return TS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
      ws_bytes < ts_topk_workspace_size(B, max_ctx, k))
    return TS_ERR_WORKSPACE;
  return TS_OK;
}

ts_status topk_enqueue(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                       int max_ctx, int k, int32_t* ids, void* ws, int32_t* err,
                       cudaStream_t stream) {
  return launch_topk(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, ws, err, stream);
}

}  // namespace dsakv

extern "C" ts_status ts_topk(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                             int max_ctx, int k, int32_t* ids, void* ws, size_t ws_bytes,
                             int32_t* err, cudaStream_t stream) {
  const ts_status st = topk_check(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, ws, ws_bytes);
  if (st != TS_OK) return st;
  return topk_enqueue(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, ws, err, stream);
}

// ---------------------------------------------------------------------------
// ts_topk_noalloc: the same top-k with its scratch in a fixed device array, for
// callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace dsakv {
namespace {

constexpr int kNoAllocMaxB = 128;
constexpr int64_t kNoAllocMaxPositions = int64_t(1) << 22;  // B * max_ctx
constexpr size_t kNoAllocScratchBytes =
    ((size_t(kNoAllocMaxB) * kBins * 4 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxB) * 8 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxPositions) * 8 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxPositions / 32 + kNoAllocMaxB) * 4 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxPositions / kChunk + kNoAllocMaxB) * 4 + 255) & ~size_t(255));

// Module-scope scratch: every device that loads the library holds it (about
// 34.5 MiB) until the process exits. Host code must not pass the symbol
// itself to a kernel; it takes the device address from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace dsakv

extern "C" ts_status ts_topk_noalloc(const float* scores, int64_t ctx_stride,
                                     const int32_t* ctx_len, int B, int max_ctx, int k,
                                     int32_t* ids, int32_t* err, cudaStream_t stream) {
  const ts_status st = check_topk_args(scores, ctx_stride, ctx_len, B, max_ctx, k, ids);
  if (st != TS_OK) return st;
  if (B > kNoAllocMaxB || int64_t(B) * max_ctx > kNoAllocMaxPositions) return TS_ERR_UNSUPPORTED;
  if (ts_topk_workspace_size(B, max_ctx, k) > kNoAllocScratchBytes) return TS_ERR_UNSUPPORTED;
  void* ws = scratch_on_current_device();
  if (!ws) return TS_ERR_CUDA;
  // every call clears what must start at zero before its kernels read it
  return launch_topk(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, ws, err, stream);
}
