// ts_topk: the k positions of largest Lightning-Indexer score per request
// (GLM-5.2 shared-Indexer KV Cache Offload, §2.1: the indexer selects the 2048
// history positions most relevant to the query, and sparse attention reads
// only those). Ties go to the lower position; output in ascending position.
//
// Radix select in three passes, many CTAs per request:
//   hist   : every CTA histograms the top 12 bits of the order-preserving
//            32-bit key of its chunk and adds it to the request's histogram.
//   select : every CTA finds the threshold bin (the bin holding the k-th
//            largest key), marks the positions of higher bins in a bitmap
//            (one 32-bit word per 32 positions, built by a warp ballot), and
//            appends the threshold bin's (key, position) pairs to a list.
//   finish : one CTA per request resolves the threshold inside that list
//            (two more 10-bit digits, then the lowest positions among exact
//            ties), sets their bits, and writes the set positions of the
//            bitmap in order: the output comes out sorted without a sort.
#include "common.cuh"

namespace dsakv {
namespace {

constexpr int kBins = 4096;          // top 12 bits of the key
constexpr int kChunk = 16384;        // positions per CTA in hist / select
constexpr int kThreads = 512;
constexpr int kFinishThreads = 1024;
constexpr int kMaxK = 8192;

struct TopkWs {
  uint32_t* hist;        // [B][kBins]
  uint32_t* cand_count;  // [B]
  uint64_t* cand;        // [B][max_ctx]  (key << 32 | position)
  uint32_t* bitmap;      // [B][words]
  int64_t words;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline TopkWs carve(void* ws, int B, int max_ctx) {
  TopkWs w;
  char* p = static_cast<char*>(ws);
  w.hist = reinterpret_cast<uint32_t*>(p);
  p += align256(size_t(B) * kBins * 4);
  w.cand_count = reinterpret_cast<uint32_t*>(p);
  p += align256(size_t(B) * 4);
  w.cand = reinterpret_cast<uint64_t*>(p);
  p += align256(size_t(B) * max_ctx * 8);
  w.bitmap = reinterpret_cast<uint32_t*>(p);
  w.words = (max_ctx + 31) / 32;
  return w;
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

// Threshold bin of the 4096-bin histogram: the bin t with
// above(t) < k <= above(t) + hist[t], above(t) = count in bins > t.
// Block-wide; every thread gets the result. smem: >= 2 * blockDim ints.
__device__ void find_threshold_bin(const uint32_t* hist, int k, int* sbuf, int* bin_out,
                                   int* above_out) {
  const int nt = blockDim.x;
  const int per = kBins / nt;  // 8 (512 threads) or 4 (1024 threads)
  const int lo = threadIdx.x * per;
  int tot = 0;
  for (int i = 0; i < per; ++i) tot += static_cast<int>(hist[lo + i]);
  // exclusive suffix sum over threads = total - inclusive prefix
  int total;
  int ex = block_exclusive_scan(tot, sbuf, &total);
  int above = total - ex - tot;  // count in bins above this thread's range
  if (threadIdx.x == 0) {
    sbuf[40] = -1;
    sbuf[41] = 0;
  }
  __syncthreads();
  int cum = above;
  for (int i = per - 1; i >= 0; --i) {
    int h = static_cast<int>(hist[lo + i]);
    if (cum < k && cum + h >= k) {
      sbuf[40] = lo + i;
      sbuf[41] = cum;
    }
    cum += h;
  }
  __syncthreads();
  *bin_out = sbuf[40];
  *above_out = sbuf[41];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const float* __restrict__ scores,
                                                             int64_t ctx_stride,
                                                             const int32_t* __restrict__ ctx_len,
                                                             int k, int max_ctx, TopkWs ws,
                                                             int32_t* err) {
  __shared__ uint32_t h[kBins];
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  if (!ctx_ok(n, k, max_ctx)) return;
  const int64_t start = int64_t(blockIdx.x) * kChunk;
  if (start >= n) return;
  const int64_t end = min(start + int64_t(kChunk), int64_t(n));
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
  __syncthreads();
  const float* row = scores + int64_t(b) * ctx_stride;
  bool nan = false;
  for (int64_t i = start + int64_t(threadIdx.x) * 4; i < end; i += int64_t(kThreads) * 4) {
    if (i + 4 <= end) {
      float4 v = __ldg(reinterpret_cast<const float4*>(row + i));
      atomicAdd(&h[score_key(v.x, nan) >> 20], 1u);
      atomicAdd(&h[score_key(v.y, nan) >> 20], 1u);
      atomicAdd(&h[score_key(v.z, nan) >> 20], 1u);
      atomicAdd(&h[score_key(v.w, nan) >> 20], 1u);
    } else {
      for (int64_t j = i; j < end; ++j) atomicAdd(&h[score_key(__ldg(row + j), nan) >> 20], 1u);
    }
  }
  if (nan) report(err, TS_DEVERR_NAN);
  __syncthreads();
  uint32_t* gh = ws.hist + int64_t(b) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (h[i]) atomicAdd(&gh[i], h[i]);
}

__global__ void __launch_bounds__(kThreads) topk_select_kernel(const float* __restrict__ scores,
                                                               int64_t ctx_stride,
                                                               const int32_t* __restrict__ ctx_len,
                                                               int k, int max_ctx, TopkWs ws) {
  __shared__ int sbuf[64];
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  if (!ctx_ok(n, k, max_ctx)) return;
  const int64_t start = int64_t(blockIdx.x) * kChunk;
  if (start >= n) return;
  int t1, above;
  find_threshold_bin(ws.hist + int64_t(b) * kBins, k, sbuf, &t1, &above);
  const int64_t end = min(start + int64_t(kChunk), int64_t(n));
  const float* row = scores + int64_t(b) * ctx_stride;
  uint32_t* bits = ws.bitmap + int64_t(b) * ws.words;
  uint64_t* cand = ws.cand + int64_t(b) * max_ctx;
  const int lane = threadIdx.x & 31;
  // each warp covers 32 consecutive positions per iteration: one bitmap word
  for (int64_t base = start + (threadIdx.x & ~31); base < end; base += kThreads) {
    const int64_t i = base + lane;
    bool nan = false;
    uint32_t key = 0;
    int bin = -1;
    if (i < end) {
      key = score_key(__ldg(row + i), nan);
      bin = static_cast<int>(key >> 20);
    }
    const uint32_t above_mask = __ballot_sync(0xffffffffu, bin > t1);
    const uint32_t tie_mask = __ballot_sync(0xffffffffu, bin == t1);
    if (lane == 0) bits[base >> 5] = above_mask;
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

// Among the candidates selected by `pred`, find the digit value t of
// (value >> shift) & (nbins-1) such that the candidates with a digit
// preferred to t number fewer than `need` and those preferred or equal
// reach it. `high_first` prefers larger digits (keys), else smaller
// (positions). Returns t and the count strictly preferred.
template <typename Pred, typename Digit>
__device__ void radix_digit(const uint64_t* cand, uint32_t c, int nbins, bool high_first, int need,
                            Pred pred, Digit digit, uint32_t* hist, int* sbuf, int* t_out,
                            int* before_out) {
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
    uint64_t e = __ldcg(cand + i);
    if (pred(e)) atomicAdd(&hist[digit(e)], 1u);
  }
  __syncthreads();
  // scan bins in preference order; nbins <= 2048 and blockDim = 1024
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  int tot = 0;
  for (int j = 0; j < per; ++j) {
    int r = threadIdx.x * per + j;  // rank in preference order
    if (r < nbins) tot += hist[high_first ? nbins - 1 - r : r];
  }
  int total;
  int ex = block_exclusive_scan(tot, sbuf, &total);
  if (threadIdx.x == 0) {
    sbuf[40] = -1;
    sbuf[41] = 0;
  }
  __syncthreads();
  int cum = ex;
  for (int j = 0; j < per; ++j) {
    int r = threadIdx.x * per + j;
    if (r >= nbins) break;
    int bin = high_first ? nbins - 1 - r : r;
    int h = hist[bin];
    if (cum < need && cum + h >= need) {
      sbuf[40] = bin;
      sbuf[41] = cum;
    }
    cum += h;
  }
  __syncthreads();
  *t_out = sbuf[40];
  *before_out = sbuf[41];
  __syncthreads();
}

__global__ void __launch_bounds__(kFinishThreads) topk_finish_kernel(
    const int32_t* __restrict__ ctx_len, int k, int max_ctx, TopkWs ws, int32_t* __restrict__ ids,
    int32_t* err) {
  __shared__ uint32_t hist[2048];
  __shared__ int sbuf[64];
  const int b = blockIdx.x;
  const int n = ctx_len[b];
  int32_t* out = ids + int64_t(b) * k;
  if (!ctx_ok(n, k, max_ctx)) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    if (threadIdx.x == 0) report(err, TS_DEVERR_CTX);
    return;
  }
  // the 12-bit threshold bin, as the select pass found it
  int t1, above1;
  {
    // find_threshold_bin wants kBins / blockDim bins per thread: 4 here
    find_threshold_bin(ws.hist + int64_t(b) * kBins, k, sbuf, &t1, &above1);
  }
  const uint64_t* cand = ws.cand + int64_t(b) * max_ctx;
  const uint32_t c = __ldcg(ws.cand_count + b);
  const int need1 = k - above1;  // >= 1 candidates to take from the list

  // digit 2: key bits [19:10]
  int t2, before2;
  radix_digit(
      cand, c, 1024, true, need1, [](uint64_t) { return true; },
      [](uint64_t e) { return static_cast<int>((e >> 42) & 1023u); }, hist, sbuf, &t2, &before2);
  const int need2 = need1 - before2;
  // digit 3: key bits [9:0] among digit-2 == t2
  int t3, before3;
  radix_digit(
      cand, c, 1024, true, need2,
      [t2](uint64_t e) { return static_cast<int>((e >> 42) & 1023u) == t2; },
      [](uint64_t e) { return static_cast<int>((e >> 32) & 1023u); }, hist, sbuf, &t3, &before3);
  const int need3 = need2 - before3;  // ties to take at the exact threshold key
  const uint32_t T = (static_cast<uint32_t>(t1) << 20) | (static_cast<uint32_t>(t2) << 10) |
                     static_cast<uint32_t>(t3);
  // lowest positions among the exact ties: three digits of the position
  auto is_tie = [T](uint64_t e) { return static_cast<uint32_t>(e >> 32) == T; };
  int pa, ba, pb, bb, pc, bc;
  radix_digit(
      cand, c, 2048, false, need3, is_tie,
      [](uint64_t e) { return static_cast<int>((static_cast<uint32_t>(e) >> 20) & 2047u); }, hist,
      sbuf, &pa, &ba);
  radix_digit(
      cand, c, 1024, false, need3 - ba,
      [is_tie, pa](uint64_t e) {
        return is_tie(e) && static_cast<int>((static_cast<uint32_t>(e) >> 20) & 2047u) == pa;
      },
      [](uint64_t e) { return static_cast<int>((static_cast<uint32_t>(e) >> 10) & 1023u); }, hist,
      sbuf, &pb, &bb);
  radix_digit(
      cand, c, 1024, false, need3 - ba - bb,
      [is_tie, pa, pb](uint64_t e) {
        const uint32_t p = static_cast<uint32_t>(e);
        return is_tie(e) && static_cast<int>((p >> 20) & 2047u) == pa &&
               static_cast<int>((p >> 10) & 1023u) == pb;
      },
      [](uint64_t e) { return static_cast<int>(static_cast<uint32_t>(e) & 1023u); }, hist, sbuf,
      &pc, &bc);
  const uint32_t cut = (static_cast<uint32_t>(pa) << 20) | (static_cast<uint32_t>(pb) << 10) |
                       static_cast<uint32_t>(pc);

  // mark the chosen candidates
  uint32_t* bits = ws.bitmap + int64_t(b) * ws.words;
  for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
    const uint64_t e = __ldcg(cand + i);
    const uint32_t key = static_cast<uint32_t>(e >> 32), pos = static_cast<uint32_t>(e);
    if (key > T || (key == T && pos <= cut)) atomicOr(bits + (pos >> 5), 1u << (pos & 31));
  }
  __syncthreads();

  // ordered write-out of the set bits
  const int64_t nwords = (n + 31) / 32;
  const int64_t per = (nwords + blockDim.x - 1) / blockDim.x;
  const int64_t w0 = int64_t(threadIdx.x) * per;
  const int64_t w1 = min(w0 + per, nwords);
  int cnt = 0;
  for (int64_t w = w0; w < w1; ++w) cnt += __popc(__ldcg(bits + w));
  int total;
  int pos = block_exclusive_scan(cnt, sbuf, &total);
  if (total != k) {
    if (threadIdx.x == 0) report(err, TS_DEVERR_COUNT);
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    return;
  }
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t m = __ldcg(bits + w);
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      out[pos++] = static_cast<int32_t>(w * 32 + bit);
    }
  }
}

}  // namespace
}  // namespace dsakv

using namespace dsakv;

extern "C" size_t ts_topk_workspace_size(int B, int max_ctx, int k) {
  (void)k;
  if (B <= 0 || max_ctx <= 0) return 0;
  const int64_t words = (int64_t(max_ctx) + 31) / 32;
  return align256(size_t(B) * kBins * 4) + align256(size_t(B) * 4) +
         align256(size_t(B) * max_ctx * 8) + align256(size_t(B) * words * 4);
}

extern "C" ts_status ts_topk(const float* scores, int64_t ctx_stride, const int32_t* ctx_len, int B,
                             int max_ctx, int k, int32_t* ids, void* ws, size_t ws_bytes,
                             int32_t* err, cudaStream_t stream) {
  if (!scores || !ctx_len || !ids || !ws) return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || max_ctx < k || ctx_stride < max_ctx) return TS_ERR_INVALID_ARG;
  if (k > kMaxK || B > 65535) return TS_ERR_UNSUPPORTED;
  if (!aligned16(scores) || (ctx_stride & 3) != 0) return TS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < ts_topk_workspace_size(B, max_ctx, k))
    return TS_ERR_WORKSPACE;
  TopkWs w = carve(ws, B, max_ctx);
  // histograms and list counters start at zero on every call
  if (cudaMemsetAsync(ws, 0, align256(size_t(B) * kBins * 4) + align256(size_t(B) * 4), stream) !=
      cudaSuccess)
    return TS_ERR_CUDA;
  const dim3 grid((max_ctx + kChunk - 1) / kChunk, B);
  topk_hist_kernel<<<grid, kThreads, 0, stream>>>(scores, ctx_stride, ctx_len, k, max_ctx, w, err);
  topk_select_kernel<<<grid, kThreads, 0, stream>>>(scores, ctx_stride, ctx_len, k, max_ctx, w);
  topk_finish_kernel<<<B, kFinishThreads, 0, stream>>>(ctx_len, k, max_ctx, w, ids, err);
  return launch_status();
}

// ---------------------------------------------------------------------------
// ts_topk_noalloc: the same top-k with its scratch in a fixed device array, for
// callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
#include <mutex>

namespace dsakv {
namespace {

constexpr int kNoAllocMaxB = 128;
constexpr int64_t kNoAllocMaxPositions = int64_t(1) << 22;  // B * max_ctx
constexpr size_t kNoAllocScratchBytes =
    ((size_t(kNoAllocMaxB) * kBins * 4 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxB) * 4 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxPositions) * 8 + 255) & ~size_t(255)) +
    ((size_t(kNoAllocMaxPositions / 32 + kNoAllocMaxB) * 4 + 255) & ~size_t(255));

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
  if (!scores || !ctx_len || !ids) return TS_ERR_INVALID_ARG;
  if (B <= 0 || k <= 0 || max_ctx < k || ctx_stride < max_ctx) return TS_ERR_INVALID_ARG;
  if (k > kMaxK || B > kNoAllocMaxB || int64_t(B) * max_ctx > kNoAllocMaxPositions)
    return TS_ERR_UNSUPPORTED;
  if (!aligned16(scores) || (ctx_stride & 3) != 0) return TS_ERR_INVALID_ARG;
  if (ts_topk_workspace_size(B, max_ctx, k) > kNoAllocScratchBytes) return TS_ERR_UNSUPPORTED;
  void* ws = scratch_on_current_device();
  if (!ws) return TS_ERR_CUDA;
  TopkWs w = carve(ws, B, max_ctx);
  // the histograms and list counters left by the previous call are cleared
  if (cudaMemsetAsync(ws, 0, align256(size_t(B) * kBins * 4) + align256(size_t(B) * 4), stream) !=
      cudaSuccess)
    return TS_ERR_CUDA;
  const dim3 grid((max_ctx + kChunk - 1) / kChunk, B);
  topk_hist_kernel<<<grid, kThreads, 0, stream>>>(scores, ctx_stride, ctx_len, k, max_ctx, w, err);
  topk_select_kernel<<<grid, kThreads, 0, stream>>>(scores, ctx_stride, ctx_len, k, max_ctx, w);
  topk_finish_kernel<<<B, kFinishThreads, 0, stream>>>(ctx_len, k, max_ctx, w, ids, err);
  return launch_status();
}
