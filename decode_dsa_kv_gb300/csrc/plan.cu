// dsa_plan: the shared plan of one IndexShare group (GLM-5.2 shared-Indexer KV
// Cache Offload, §4.2 shared planning and §5 DsaPlan; pool policy §4.3).
//
// One CTA per request. The request's pool tags are staged in shared memory;
// every selected id is looked up in the W ways of its set (token mod S); the
// misses are compacted in ascending id (warp ballots + a block scan when the
// ids arrive sorted and distinct, a shared-memory bitonic sort otherwise),
// counted per set, bucketed by set, and ranked inside their set to get the
// FIFO victim slot and whether the miss survives a same-step overflow.
#include <climits>

#include "common.cuh"
#include "ops.h"

namespace dsakv {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxK = 4096;
constexpr size_t kMaxSmem = 200 * 1024;

struct PlanSmem {
  int* tags;      // [P]
  int* cnt;       // [S]  misses per set
  int* off;       // [S]  exclusive prefix of cnt
  int* fill;      // [S]  bucket fill counters
  int* mids;      // [k]  miss ids, ascending
  int* mpos;      // [k]  first position of each miss
  int* bucket;    // [k]  miss ids grouped by set
  int* src;       // [k]  this request's src_map
  uint64_t* key;  // [pow2(k)] sort keys (general path)
  int* scratch;   // [64]
  int* flags;     // [4]
  uint32_t* hit;  // [ceil(P / 32)] slots read as hits in this step
};

__host__ __device__ inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// sort keys first (8-byte entries, at least 16 bytes so the int region that
// follows stays 16-byte aligned for the int4 tag reads)
__host__ __device__ inline size_t key_bytes(int k) {
  return size_t(pow2_at_least(k < 2 ? 2 : k)) * 8;
}

__host__ __device__ inline size_t plan_smem_bytes(int P, int S, int k) {
  return key_bytes(k) + size_t(P) * 4 + size_t(S) * 12 + size_t(k) * 16 + 64 * 4 + 4 * 4 +
         size_t((P + 31) / 32) * 4 + 64;
}

__device__ PlanSmem carve(char* base, int P, int S, int k) {
  PlanSmem s;
  uint64_t* key = reinterpret_cast<uint64_t*>(base);  // 8-byte aligned first
  s.key = key;
  int* p = reinterpret_cast<int*>(base + key_bytes(k));
  s.tags = p;
  p += P;
  s.cnt = p;
  p += S;
  s.off = p;
  p += S;
  s.fill = p;
  p += S;
  s.mids = p;
  p += k;
  s.mpos = p;
  p += k;
  s.bucket = p;
  p += k;
  s.src = p;
  p += k;
  s.scratch = p;
  p += 64;
  s.flags = p;
  p += 4;
  s.hit = reinterpret_cast<uint32_t*>(p);
  return s;
}

// Lowest way of set `set` whose tag equals t, or -1.
__device__ __forceinline__ int lookup(const int* tags, int set, int W, int t) {
  const int* row = tags + set * W;
  if ((W & 3) == 0) {
    for (int w = 0; w < W; w += 4) {
      int4 v = *reinterpret_cast<const int4*>(row + w);
      if (v.x == t) return w;
      if (v.y == t) return w + 1;
      if (v.z == t) return w + 2;
      if (v.w == t) return w + 3;
    }
    return -1;
  }
  for (int w = 0; w < W; ++w)
    if (row[w] == t) return w;
  return -1;
}

__global__ void __launch_bounds__(kThreads) dsa_plan_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ ctx_len, int k,
    const int32_t* __restrict__ pool_tags, const int32_t* __restrict__ fifo_ptr, int S, int W,
    int32_t* __restrict__ src_map, int32_t* __restrict__ miss_ids, int32_t* __restrict__ miss_pos,
    int32_t* __restrict__ victim, uint8_t* __restrict__ install, int32_t* __restrict__ miss_count,
    int32_t* __restrict__ miss_rows, int32_t* __restrict__ ptr_next, int32_t* err) {
  extern __shared__ __align__(16) char smem_raw[];
  const int P = S * W;
  PlanSmem sm = carve(smem_raw, P, S, k);
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = ctx_len[b];
  const int32_t* id_row = ids + int64_t(b) * k;
  const int32_t* tag_row = pool_tags + int64_t(b) * P;
  const int32_t* ptr_row = fifo_ptr + int64_t(b) * S;

  // stage tags, clear per-set counters
  if ((P & 3) == 0 && aligned16(tag_row)) {
    for (int i = tid; i < P / 4; i += kThreads)
      reinterpret_cast<int4*>(sm.tags)[i] = __ldg(reinterpret_cast<const int4*>(tag_row) + i);
  } else {
    for (int i = tid; i < P; i += kThreads) sm.tags[i] = __ldg(tag_row + i);
  }
  for (int s = tid; s < S; s += kThreads) {
    sm.cnt[s] = 0;
    sm.fill[s] = 0;
    const int p = ptr_row[s];
    if (p < 0 || p >= W) report(err, TS_DEVERR_PTR_RANGE);
  }
  for (int i = tid; i < (P + 31) / 32; i += kThreads) sm.hit[i] = 0;
  __syncthreads();

  // classify, and check whether the ids are strictly ascending
  bool ascending = true;
  bool bad_id = false;
  for (int j = tid; j < k; j += kThreads) {
    const int t = id_row[j];
    if (j + 1 < k && !(t < id_row[j + 1])) ascending = false;
    int src;
    if (t < 0 || t >= n) {
      src = INT_MIN;
      bad_id = true;
    } else {
      const int set = t % S;
      const int way = lookup(sm.tags, set, W, t);
      src = way >= 0 ? set * W + way : -1 - t;
      if (way >= 0) atomicOr(sm.hit + (src >> 5), 1u << (src & 31));
    }
    src_map[int64_t(b) * k + j] = src;
    sm.src[j] = src;
  }
  if (bad_id) report(err, TS_DEVERR_ID_RANGE);
  ascending = __syncthreads_and(ascending);
  {
    // positions that miss, repeats included
    int c = 0;
    for (int j = tid; j < k; j += kThreads) c += (sm.src[j] < 0 && sm.src[j] != INT_MIN);
    int total;
    block_exclusive_scan(c, sm.scratch, &total);
    if (tid == 0) miss_rows[b] = total;
  }

  int M;
  if (ascending) {
    // misses in position order are already ascending and distinct: an
    // ordered compaction. Each thread owns a contiguous run of positions.
    const int per = (k + kThreads - 1) / kThreads;
    const int j0 = tid * per, j1 = min(j0 + per, k);
    int c = 0;
    for (int j = j0; j < j1; ++j) {
      const int src = sm.src[j];
      c += (src < 0 && src != INT_MIN);
    }
    int total;
    int o = block_exclusive_scan(c, sm.scratch, &total);
    for (int j = j0; j < j1; ++j) {
      const int src = sm.src[j];
      if (src < 0 && src != INT_MIN) {
        sm.mids[o] = -1 - src;
        sm.mpos[o] = j;
        ++o;
      }
    }
    M = total;
  } else {
    // general ids: sort (id, position) pairs of the misses, keep the first of
    // every id
    const int np2 = pow2_at_least(k);
    for (int j = tid; j < np2; j += kThreads) {
      uint64_t key = ~0ull;
      if (j < k) {
        const int src = sm.src[j];
        if (src < 0 && src != INT_MIN)
          key = (static_cast<uint64_t>(static_cast<uint32_t>(-1 - src)) << 32) | uint32_t(j);
      }
      sm.key[j] = key;
    }
    __syncthreads();
    for (int size = 2; size <= np2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < np2 / 2; i += kThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const uint64_t a = sm.key[lo], c2 = sm.key[hi];
          if ((a > c2) == up) {
            sm.key[lo] = c2;
            sm.key[hi] = a;
          }
        }
        __syncthreads();
      }
    }
    const int per = (np2 + kThreads - 1) / kThreads;
    const int j0 = tid * per, j1 = min(j0 + per, np2);
    auto keep = [&](int j) {
      const uint64_t e = sm.key[j];
      if (e == ~0ull) return false;
      return j == 0 || (sm.key[j - 1] >> 32) != (e >> 32);
    };
    int c = 0;
    for (int j = j0; j < j1; ++j) c += keep(j);
    int total;
    int o = block_exclusive_scan(c, sm.scratch, &total);
    for (int j = j0; j < j1; ++j) {
      if (keep(j)) {
        sm.mids[o] = static_cast<int>(sm.key[j] >> 32);
        sm.mpos[o] = static_cast<int>(sm.key[j] & 0xffffffffu);
        ++o;
      }
    }
    M = total;
  }
  __syncthreads();

  // misses per set, set offsets, buckets
  for (int i = tid; i < M; i += kThreads) atomicAdd(&sm.cnt[sm.mids[i] % S], 1);
  __syncthreads();
  {
    const int per = (S + kThreads - 1) / kThreads;
    const int s0 = tid * per, s1 = min(s0 + per, S);
    int c = 0;
    for (int s = s0; s < s1; ++s) c += sm.cnt[s];
    int total;
    int o = block_exclusive_scan(c, sm.scratch, &total);
    for (int s = s0; s < s1; ++s) {
      sm.off[s] = o;
      o += sm.cnt[s];
    }
  }
  __syncthreads();
  for (int i = tid; i < M; i += kThreads) {
    const int t = sm.mids[i], set = t % S;
    sm.bucket[sm.off[set] + atomicAdd(&sm.fill[set], 1)] = t;
  }
  __syncthreads();

  // rank inside the set (ascending id) -> victim slot and survival
  for (int i = tid; i < M; i += kThreads) {
    const int t = sm.mids[i], set = t % S;
    const int c = sm.cnt[set], o = sm.off[set];
    int r = 0;
    for (int e = 0; e < c; ++e) r += sm.bucket[o + e] < t;
    const int p = ptr_row[set];
    const int pp = (p >= 0 && p < W) ? p : 0;
    const int64_t g = int64_t(b) * k + i;
    miss_ids[g] = t;
    miss_pos[g] = sm.mpos[i];
    victim[g] = set * W + (pp + r) % W;
    // 1: the victim slot is read by no position of this step, the row may
    // go in on arrival; 2: it is read as a hit, the row goes in after the
    // layer's reads ([GLM] §4.4)
    const int v = set * W + (pp + r) % W;
    install[g] = r >= c - W ? ((sm.hit[v >> 5] >> (v & 31)) & 1u ? 2 : 1) : 0;
  }
  for (int s = tid; s < S; s += kThreads) {
    const int p = ptr_row[s];
    const int pp = (p >= 0 && p < W) ? p : 0;
    ptr_next[int64_t(b) * S + s] = (pp + sm.cnt[s]) % W;
  }
  if (tid == 0) miss_count[b] = M;
}

// ---------------------------------------------------------------------------
// dsa_plan_reuse: the base design's adjacent-step reuse (GLM-5.2 shared-Indexer
// KV Cache Offload, §2.1 GatherSelectionKvCache and §2.2): a token the
// previous step also selected is served from the previous step's selection
// buffer (its row there = its position in the previous ids), any other token
// from host memory. One CTA per request: the previous ids in shared memory,
// a binary search per position, the misses compacted in position order (which
// is ascending id) by a block scan.
// ---------------------------------------------------------------------------
constexpr int kReuseThreads = 1024;

__global__ void __launch_bounds__(kReuseThreads) dsa_plan_reuse_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ prev_ids,
    const int32_t* __restrict__ ctx_len, int k, int32_t* __restrict__ src_map,
    int32_t* __restrict__ miss_ids, int32_t* __restrict__ miss_pos,
    int32_t* __restrict__ miss_count, int32_t* __restrict__ miss_rows, int32_t* err) {
  extern __shared__ int prev[];  // [k], then 64 ints of scan scratch
  int* scratch = prev + k;
  const int b = blockIdx.x;
  const int n = ctx_len[b];
  const int32_t* id = ids + int64_t(b) * k;
  for (int i = threadIdx.x; i < k; i += kReuseThreads) prev[i] = prev_ids[int64_t(b) * k + i];
  __syncthreads();
  // each thread a contiguous run of positions, so that the scan keeps order
  const int per = (k + kReuseThreads - 1) / kReuseThreads;
  const int j0 = threadIdx.x * per, j1 = min(j0 + per, k);
  int bad = 0, misses = 0;
  for (int j = j0; j < j1; ++j) {
    const int t = id[j];
    if (j > 0 && id[j - 1] >= t) bad |= TS_DEVERR_ORDER;
    if (j > 0 && prev[j] >= 0 && prev[j - 1] >= prev[j]) bad |= TS_DEVERR_ORDER;
    if (t < 0 || t >= n) {
      bad |= TS_DEVERR_ID_RANGE;
      src_map[int64_t(b) * k + j] = INT_MIN;
      continue;
    }
    int lo = 0, hi = k;  // first entry >= t (empty entries, -1, sort first)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (prev[mid] < t) lo = mid + 1;
      else hi = mid;
    }
    const bool hit = lo < k && prev[lo] == t;
    src_map[int64_t(b) * k + j] = hit ? lo : -1 - t;
    misses += hit ? 0 : 1;
  }
  int total;
  int at = block_exclusive_scan(misses, scratch, &total);
  for (int j = j0; j < j1; ++j) {
    const int s = src_map[int64_t(b) * k + j];
    if (s < 0 && s != INT_MIN) {
      miss_ids[int64_t(b) * k + at] = -1 - s;
      miss_pos[int64_t(b) * k + at] = j;
      ++at;
    }
  }
  if (threadIdx.x == 0) {
    miss_count[b] = total;
    miss_rows[b] = total;  // ascending ids: no token repeats
  }
  if (bad) report(err, bad);
}

// ---------------------------------------------------------------------------
// dsa_plan_lru: the fully associative LRU pool (GLM-5.2 shared-Indexer KV Cache
// Offload, §3: the 8192-entry device pool the pages built before the
// set-associative FIFO). Same outputs as dsa_plan, plus the pool's metadata
// updated in place. The policy: the step's hits are touched in position
// order, then its misses are installed in ascending id, each into the least
// recently used slot (empty slots first, lowest index first).
//
// The metadata is the slots' recency order itself (lru_order, least recently
// used first) rather than a clock and per-slot stamps, so no plan sorts: with
// k <= P a step misses at most as many tokens as it has slots it does not hit,
// so its victims are the first M of those slots in the old order, and the
// new order is
//     [slots neither hit nor evicted, old order] ++ [hit slots, position order]
//     ++ [victims, install order]
// (the touched hits are more recent than anything untouched, the installs
// more recent than the hits). A cold pool is all empty with the identity
// order, which lists the empty slots first in index order, and every step
// keeps them so. One CTA per request: every slot's tag is looked up in the
// (ascending) selected ids by binary search; two block-wide scans place the
// hits (over positions) and the slots not hit (over the old order).
// ---------------------------------------------------------------------------
constexpr int kLruThreads = 1024;

__host__ __device__ inline size_t lru_smem_bytes(int P, int k) {
  // old order [P] int; hit flags [P] bytes; seen bitmap [P/32] words;
  // ids, hit slots, miss ids [k] ints each; scan scratch
  return size_t(P) * 4 + ((size_t(P) + 15) & ~size_t(15)) + size_t((P + 31) / 32) * 4 +
         size_t(k) * 12 + 64 * 4 + 16;
}

__device__ __forceinline__ int find_sorted(const int* v, int n, int t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < t) lo = mid + 1;
    else hi = mid;
  }
  return (lo < n && v[lo] == t) ? lo : -1;
}

__global__ void __launch_bounds__(kLruThreads) dsa_plan_lru_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ ctx_len, int k,
    int32_t* __restrict__ pool_tags, int32_t* __restrict__ lru_order, int P,
    int32_t* __restrict__ src_map, int32_t* __restrict__ miss_ids,
    int32_t* __restrict__ miss_pos, int32_t* __restrict__ victim,
    uint8_t* __restrict__ install, int32_t* __restrict__ miss_count,
    int32_t* __restrict__ miss_rows, int32_t* err) {
  extern __shared__ __align__(16) char smem_raw[];
  int* order_s = reinterpret_cast<int*>(smem_raw);                              // [P]
  uint8_t* hit_s = reinterpret_cast<uint8_t*>(order_s + P);                     // [P]
  uint32_t* seen = reinterpret_cast<uint32_t*>(hit_s + ((P + 15) & ~15));       // [P/32]
  int* id_s = reinterpret_cast<int*>(seen + (P + 31) / 32);                     // [k]
  int* src_s = id_s + k;                                                        // [k]
  int* mid_s = src_s + k;                                                       // [k]
  int* scratch = mid_s + k;                                                     // [64]
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = ctx_len[b];
  const int32_t* id_row = ids + int64_t(b) * k;
  int32_t* tag_row = pool_tags + int64_t(b) * P;
  int32_t* order_row = lru_order + int64_t(b) * P;

  bool ascending = true, bad_id = false;
  for (int j = tid; j < k; j += kLruThreads) {
    const int t = id_row[j];
    if (j + 1 < k && !(t < id_row[j + 1])) ascending = false;
    if (t < 0 || t >= n) bad_id = true;
    id_s[j] = t;
    src_s[j] = -1;
  }
  for (int w = tid; w < (P + 31) / 32; w += kLruThreads) seen[w] = 0;
  if (bad_id) report(err, TS_DEVERR_ID_RANGE);
  ascending = __syncthreads_and(ascending);
  if (!ascending && tid == 0) report(err, TS_DEVERR_ORDER);

  // the old order (a permutation of the slots), and every slot's hit position
  bool bad_order = false;
  int hit_slots = 0;
  for (int i = tid; i < P; i += kLruThreads) {
    int s = order_row[i];
    if (s < 0 || s >= P) {
      bad_order = true;
      s = 0;
    } else if (atomicOr(seen + (s >> 5), 1u << (s & 31)) & (1u << (s & 31))) {
      bad_order = true;
    }
    order_s[i] = s;
    const int t = tag_row[i];
    const int j = t >= 0 ? find_sorted(id_s, k, t) : -1;
    if (j >= 0) {
      src_s[j] = i;
      ++hit_slots;
    }
    hit_s[i] = j >= 0;
  }
  bad_order = __syncthreads_or(bad_order);

  // source map; hits placed in position order after the untouched slots;
  // misses compacted in position order, which is ascending id. Each thread
  // owns a contiguous run of positions.
  const int per = (k + kLruThreads - 1) / kLruThreads;
  const int j0 = min(tid * per, k), j1 = min(j0 + per, k);
  int nh = 0, nm = 0;
  for (int j = j0; j < j1; ++j) {
    const int t = id_s[j];
    if (src_s[j] >= 0) ++nh;
    else if (t >= 0 && t < n) ++nm;
  }
  int H, M, HS;
  int h = block_exclusive_scan(nh, scratch, &H);
  int mi = block_exclusive_scan(nm, scratch, &M);
  block_exclusive_scan(hit_slots, scratch, &HS);
  // a token held by two slots, or an order that is not a permutation of the
  // slots: the pool's metadata is corrupt (the plan is then undefined)
  const bool corrupt = bad_order || HS != H;
  if (corrupt && tid == 0) report(err, TS_DEVERR_SLOT_RANGE);
  for (int j = j0; j < j1; ++j) {
    const int t = id_s[j];
    const int slot = src_s[j];
    int src;
    if (slot >= 0) {
      src = slot;
      if (!corrupt) order_row[P - M - H + h] = slot;
      ++h;
    } else if (t >= 0 && t < n) {
      src = -1 - t;
      mid_s[mi] = t;
      miss_ids[int64_t(b) * k + mi] = t;
      miss_pos[int64_t(b) * k + mi] = j;
      ++mi;
    } else {
      src = INT_MIN;
    }
    src_map[int64_t(b) * k + j] = src;
  }

  // the slots no position hits, in the old order: the first M are the
  // victims (least recently used first), the rest move to the front
  const int per2 = (P + kLruThreads - 1) / kLruThreads;
  const int i0 = min(tid * per2, P), i1 = min(i0 + per2, P);
  int nn = 0;
  for (int i = i0; i < i1; ++i) nn += hit_s[order_s[i]] ? 0 : 1;
  int NH;
  int r = block_exclusive_scan(nn, scratch, &NH);  // (a barrier: mid_s is complete)
  for (int i = i0; i < i1; ++i) {
    const int s = order_s[i];
    if (hit_s[s]) continue;
    if (r < M) {
      const int64_t g = int64_t(b) * k + r;
      if (corrupt) {
        victim[g] = 0;
        install[g] = 0;
      } else {
        victim[g] = s;
        install[g] = 1;
        tag_row[s] = mid_s[r];
        order_row[P - M + r] = s;
      }
    } else if (!corrupt) {
      order_row[r - M] = s;
    }
    ++r;
  }
  if (corrupt)  // (victims past the slots not hit: only with corrupt metadata)
    for (int i = NH + tid; i < M; i += kLruThreads) {
      victim[int64_t(b) * k + i] = 0;
      install[int64_t(b) * k + i] = 0;
    }
  if (tid == 0) {
    miss_count[b] = M;
    miss_rows[b] = M;
  }
}

}  // namespace
}  // namespace dsakv

using namespace dsakv;

namespace dsakv {

ts_status plan_check(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                     const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                     int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos, int32_t* victim,
                     uint8_t* install, int32_t* miss_count, int32_t* miss_rows,
                     int32_t* ptr_next) {
  if (!ids || !ctx_len || !pool_tags || !fifo_ptr || !src_map || !miss_ids || !miss_pos ||
      !victim || !install || !miss_count || !miss_rows || !ptr_next)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || S <= 0 || W <= 0) return TS_ERR_INVALID_ARG;
  if (W > 32 || k > kMaxK || B > 2147483647 / 2) return TS_ERR_UNSUPPORTED;
  if (int64_t(S) * W > (1 << 24)) return TS_ERR_UNSUPPORTED;
  if (plan_smem_bytes(S * W, S, k) > kMaxSmem) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

ts_status plan_enqueue(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                       const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                       int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos, int32_t* victim,
                       uint8_t* install, int32_t* miss_count, int32_t* miss_rows,
                       int32_t* ptr_next, int32_t* err, cudaStream_t stream) {
  const size_t smem = plan_smem_bytes(S * W, S, k);
  if (cudaFuncSetAttribute(dsa_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem)) != cudaSuccess)
    return TS_ERR_CUDA;
  dsa_plan_kernel<<<B, kThreads, smem, stream>>>(ids, ctx_len, k, pool_tags, fifo_ptr, S, W,
                                                 src_map, miss_ids, miss_pos, victim, install,
                                                 miss_count, miss_rows, ptr_next, err);
  return launch_status();
}

}  // namespace dsakv

extern "C" ts_status dsa_plan(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                              const int32_t* pool_tags, const int32_t* fifo_ptr, int S, int W,
                              int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                              int32_t* victim, uint8_t* install, int32_t* miss_count,
                              int32_t* miss_rows, int32_t* ptr_next, int32_t* err,
                              cudaStream_t stream) {
  const ts_status st = dsakv::plan_check(ids, ctx_len, B, k, pool_tags, fifo_ptr, S, W, src_map,
                                         miss_ids, miss_pos, victim, install, miss_count,
                                         miss_rows, ptr_next);
  if (st != TS_OK) return st;
  return dsakv::plan_enqueue(ids, ctx_len, B, k, pool_tags, fifo_ptr, S, W, src_map, miss_ids,
                             miss_pos, victim, install, miss_count, miss_rows, ptr_next, err,
                             stream);
}

namespace dsakv {

ts_status plan_reuse_check(const int32_t* ids, const int32_t* prev_ids, const int32_t* ctx_len,
                           int B, int k, int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                           int32_t* miss_count, int32_t* miss_rows) {
  if (!ids || !prev_ids || !ctx_len || !src_map || !miss_ids || !miss_pos || !miss_count ||
      !miss_rows)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0) return TS_ERR_INVALID_ARG;
  if (k > 16384) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

ts_status plan_reuse_enqueue(const int32_t* ids, const int32_t* prev_ids, const int32_t* ctx_len,
                             int B, int k, int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                             int32_t* miss_count, int32_t* miss_rows, int32_t* err,
                             cudaStream_t stream) {
  const size_t smem = size_t(k) * 4 + 64 * 4;
  if (cudaFuncSetAttribute(dsa_plan_reuse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem)) != cudaSuccess)
    return TS_ERR_CUDA;
  dsa_plan_reuse_kernel<<<B, kReuseThreads, smem, stream>>>(ids, prev_ids, ctx_len, k, src_map,
                                                            miss_ids, miss_pos, miss_count,
                                                            miss_rows, err);
  return launch_status();
}

}  // namespace dsakv

extern "C" ts_status dsa_plan_reuse(const int32_t* ids, const int32_t* prev_ids,
                                    const int32_t* ctx_len, int B, int k, int32_t* src_map,
                                    int32_t* miss_ids, int32_t* miss_pos, int32_t* miss_count,
                                    int32_t* miss_rows, int32_t* err, cudaStream_t stream) {
  const ts_status st = dsakv::plan_reuse_check(ids, prev_ids, ctx_len, B, k, src_map, miss_ids,
                                               miss_pos, miss_count, miss_rows);
  if (st != TS_OK) return st;
  return dsakv::plan_reuse_enqueue(ids, prev_ids, ctx_len, B, k, src_map, miss_ids, miss_pos,
                                   miss_count, miss_rows, err, stream);
}

namespace dsakv {

ts_status plan_lru_check(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                         const int32_t* pool_tags, const int32_t* lru_order, int P,
                         int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                         int32_t* victim, uint8_t* install,
                         int32_t* miss_count, int32_t* miss_rows) {
  if (!ids || !ctx_len || !pool_tags || !lru_order || !src_map || !miss_ids ||
      !miss_pos || !victim || !install || !miss_count || !miss_rows)
    return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || P <= 0 || B > 65535) return TS_ERR_INVALID_ARG;
  if (k > P || k > kMaxK || lru_smem_bytes(P, k) > kMaxSmem) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

ts_status plan_lru_enqueue(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                           int32_t* pool_tags, int32_t* lru_order, int P, int32_t* src_map,
                           int32_t* miss_ids, int32_t* miss_pos, int32_t* victim, uint8_t* install, int32_t* miss_count,
                           int32_t* miss_rows, int32_t* err, cudaStream_t stream) {
  const size_t smem = lru_smem_bytes(P, k);
  static std::atomic<uint64_t> smem_set{0};
  if (!raise_smem_limit(reinterpret_cast<const void*>(dsa_plan_lru_kernel),
                        static_cast<int>(kMaxSmem), smem_set))
    return TS_ERR_CUDA;
  dsa_plan_lru_kernel<<<B, kLruThreads, smem, stream>>>(ids, ctx_len, k, pool_tags, lru_order,
                                                        P, src_map, miss_ids, miss_pos, victim,
                                                        install, miss_count, miss_rows, err);
  return launch_status();
}

}  // namespace dsakv

extern "C" ts_status dsa_plan_lru(const int32_t* ids, const int32_t* ctx_len, int B, int k,
                                  int32_t* pool_tags, int32_t* lru_order, int P,
                                  int32_t* src_map, int32_t* miss_ids, int32_t* miss_pos,
                                  int32_t* victim, uint8_t* install, int32_t* miss_count,
                                  int32_t* miss_rows, int32_t* err, cudaStream_t stream) {
  const ts_status st = dsakv::plan_lru_check(ids, ctx_len, B, k, pool_tags, lru_order, P,
                                             src_map, miss_ids, miss_pos, victim, install,
                                             miss_count, miss_rows);
  if (st != TS_OK) return st;
  return dsakv::plan_lru_enqueue(ids, ctx_len, B, k, pool_tags, lru_order, P, src_map,
                                 miss_ids, miss_pos, victim, install, miss_count, miss_rows, err,
                                 stream);
}
