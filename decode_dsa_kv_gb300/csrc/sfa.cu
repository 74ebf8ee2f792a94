// sfa_mla_decode: sparse absorbed-MLA decode attention over the selected rows
// (GLM-5.2 shared-Indexer KV Cache Offload, §2.1: SFA runs only over the
// 2048 rows the indexer selected; TokenSpeed engine audit, MLA section: one
// latent row of 512 latent + 64 rope values is both K and V, and decode is
// split over the KV rows with fp32 partials merged by log-sum-exp).
//
// One CTA per (request b, head tile of 128 heads, chunk of 512 selected rows),
// on the 5th-generation tensor cores:
//   warp 0   : TMA producer (one thread): Q and K tiles for the score product
//              (two 256-row halves) through 4 slots of 48 KB (two of them in
//              the P tile's space, free until the softmax), then V tiles for
//              the value product through 3 slots of 32 KB (128-byte swizzle).
//   warp 1   : allocates 512 TMEM columns; one thread issues tcgen05.mma.
//   warps 2-9: softmax and epilogue; two threads per head (TMEM lane), each
//              with half of the chunk's columns.
// Steps inside the CTA:
//   S[128 x 512] = Q[128 x 576] K[512 x 576]^T   -> all 512 TMEM columns
//   p = exp2(S*scale*log2e - max)  rounded to bf16, written to shared memory
//       in the K-major 128-byte-swizzled layout the MMA reads
//   O[:, 0:256]   = P V[:, 0:256]    -> TMEM columns 256..511
//   O[:, 256:512] = P V[:, 256:512]  -> TMEM columns 0..255 (S is dead by then:
//       P holds it, bf16, in shared memory)
//   O (unnormalised) -> fp32 workspace straight from TMEM, as a dim-major
//       tile [512][128 heads] (coalesced stores); the row max and the row sum
//       beside it.
// A second kernel merges the chunks of a request: out = sum_c w_c O_c /
// sum_c w_c l_c with w_c = exp2(m_c - max_c m_c). (Merging inside a cluster
// of the chunk CTAs through distributed shared memory instead measured
// slower on GB300: 45 vs 37 us a layer at the decode_batch shape alone, and
// slower in the step; the cluster waits for its slowest chunk.)
#include <climits>
#include <cmath>

#include "common.cuh"
#include "ops.h"

namespace dsakv {
namespace {

constexpr int kHeads = 128;  // MMA M
constexpr int kChunk = 512;  // rows per CTA: two score MMAs of N = 256, K of the value product
constexpr int kHalfRows = 256;
constexpr int kKB = 9;       // 64-wide blocks of the 576 dims
constexpr int kStages = 2;   // 48 KB slots of the ring region
constexpr int kSSlots = 4;   // score-phase slots: the ring's two and two in the P region
constexpr int kVSlots = 3;   // value-phase slots: 32 KB each in the ring region
constexpr uint32_t kQBytes = kHeads * 128;           // 128 heads x 64 dims
constexpr uint32_t kKBytes = kHalfRows * 128;        // 256 rows x 64 dims
constexpr uint32_t kStageBytes = kQBytes + kKBytes;  // 48 KB
constexpr uint32_t kVBox = 64 * 128;                 // 64 rows x 64 dims
constexpr uint32_t kVBytes = 4 * kVBox;              // 64 rows x 256 dims
constexpr uint32_t kPBlock = kHeads * 128;           // 128 heads x 64 rows
constexpr uint32_t kPBytes = 8 * kPBlock;            // 128 heads x 512 rows
constexpr int kScoreLoads = 2 * kKB;                 // 18 score stages
constexpr int kLoads = kScoreLoads + 16;             // + 16 value stages (8 row blocks x 2 halves)
constexpr int kSoftmaxThreads = 256;                 // warps 2..9
constexpr int kThreads = 64 + kSoftmaxThreads;
// The pool variant loads its tiles with 16-byte cp.async copies from eight
// loader warps (warp 0 and warps 10..16): 256 threads. Measured on GB300 (L2
// flushed, 128 heads x 2048 rows): 51.9 -> 45.7 us a layer at 8 requests and
// 198.6 -> 184.2 us at 128 against four loader warps (the copies' issue rate
// bounded the CTA; with 544 threads the kernel fits in 88 registers).
constexpr int kLoaderThreads = 256;
constexpr int kPoolThreads = kThreads + kLoaderThreads - 32;
constexpr uint32_t kBarBytes = 704;
// barriers first, then the 1024-byte aligned tiles (worst-case padding
// included). The total leaves room on the SM for a 0-byte CTA of another
// kernel (each CTA also holds 1 KB of reserved shared memory), so a gather or
// refill CTA can run beside an attention CTA.
constexpr uint32_t kTileBytes = kPBytes + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kBarBytes + 1024 + kTileBytes;
// The variant that reads from the pool also keeps the chunk's 512 pool rows
// (relative to the request, so P + k <= 65536) after the barrier block; it
// then fills the SM's shared memory, with no room left for another CTA.
constexpr uint32_t kRowIdxBytes = kChunk * 2;
constexpr uint32_t kPoolSmemBytes = kSmemBytes + kRowIdxBytes;
static_assert(kPoolSmemBytes <= 227 * 1024, "dynamic shared memory of one CTA");
constexpr uint64_t kWaitLimit = 2000000000ull;  // 2 s of global timer per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// 228 KB of shared memory per SM; 1 KB reserved per CTA
static_assert(kSmemBytes + 1024 + 1024 <= 228 * 1024, "room for a second, shared-memory-free CTA");

struct Bars {
  uint64_t full[kSSlots];
  uint64_t empty[kSSlots];
  uint64_t vfull[kVSlots];
  uint64_t vempty[kVSlots];
  uint64_t s_half;  // score product of the first 256 rows complete
  uint64_t s_full;
  uint64_t p_hi;    // P of rows 256..511 written (their S columns read)
  uint64_t p_lo;    // P of rows 0..255 written
  uint64_t o_half;  // value product of dims 0..255 complete
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  int issued;
  float red[kHeads];  // exchange between a head's two threads: row max, then row sum
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block");

// Wait by lane 0 of the warp, result shared by the whole warp (which is then
// converged for the .sync.aligned tcgen05 instructions that follow).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, limit_ns) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Barrier among the softmax warps only (named barrier 1, 256 threads).
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// 2^x on the special-function unit (relative error far below the bf16
// rounding the weights then get).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Where the variant that reads straight from the pool finds a selected row:
// the plan's source map over a staged-layout pool tensor, `prow` = P + k rows
// per request (the P slots, then the step's missed rows staged at P + their
// first position).
struct PoolSrc {
  const int32_t* src_map;
  const int32_t* miss_ids;
  const int32_t* miss_pos;
  const int32_t* miss_count;
  const int32_t* miss_rows;
  const uint8_t* rows;  // the pool tensor, [B][prow][576] bf16
  const uint8_t* q;     // the queries, [B][H][576] bf16
  int P, prow;
  // streamed: request b's loaders start once arrived[b] reaches its miss
  // count (the gather still running counts the staged rows in); they give up
  // when *gather_failed is set. Null: the rows are all in at launch.
  const uint32_t* arrived;
  const uint32_t* gather_failed;
  // optional: every CTA adds one as it starts (so the next layer's attention
  // can be launched once all of this launch's CTAs hold their SMs)
  uint32_t* started;
};

// 16-byte copies global -> shared that write shared memory as they land
// (cp.async, cached in L2 only); wait_group<0> waits for all of them.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Barrier among the pool variant's loader warps (named barrier 2).
__device__ __forceinline__ void loader_sync() {
  asm volatile("bar.sync 2, 256;" ::: "memory");
}

// Row of request b's part of the pool tensor that position j reads: a hit's
// slot, a miss's staged row (its first position's, when the request repeats
// tokens). A bad entry sets bits of `bad` and reads the position's own staged
// row instead (in bounds; the result is undefined).
__device__ __forceinline__ int pool_row(const PoolSrc& ps, int b, int k, int j, int M,
                                        bool repeats, int& bad) {
  const int src = __ldg(ps.src_map + int64_t(b) * k + j);
  int rel = ps.P + j;
  if (src >= 0) {
    if (src < ps.P) rel = src;
    else bad |= TS_DEVERR_SLOT_RANGE;
  } else if (src == INT_MIN) {
    bad |= TS_DEVERR_ID_RANGE;
  } else if (repeats) {
    const int f = miss_first_pos(ps.miss_ids + int64_t(b) * k, ps.miss_pos + int64_t(b) * k, M,
                                 -1 - src);
    if (f >= 0 && f < k) rel = ps.P + f;
    else bad |= TS_DEVERR_ID_RANGE;
  }
  return rel;
}

// O, the row max and the row sum of the chunk go to the workspace for
// sfa_combine_kernel. kPool = false: the rows are the selection buffer's, loaded as TMA tiles
// (tm_q, tm_k, tm_v). kPool = true: the rows are read straight from a
// staged-layout pool by the plan (`ps`), by eight loader warps with 16-byte
// cp.async copies (the maps are unused). Measured on GB300: TMA 4-row gathers
// (one instruction per 4 rows x 64 dims) kept the attention at 117 us a layer
// at the decode_batch shape against 46 us for tile loads; the TMA unit's
// instruction rate, not the memory, bounded it.
template <bool kPool>
__global__ void __launch_bounds__(kPool ? kPoolThreads : kThreads, 1)
    sfa_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, int H, int k, int HG, int C,
                     float scale_log2, float* __restrict__ opart, float2* __restrict__ ml,
                     uint64_t wait_ns, const PoolSrc ps, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Bars* bars = reinterpret_cast<Bars*>(smem_raw);
  uint16_t* ridx = reinterpret_cast<uint16_t*>(smem_raw + kBarBytes);  // kPool only
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + kBarBytes + (kPool ? kRowIdxBytes : 0u) + 1023) &
      ~uintptr_t(1023));
  uint8_t* p_tile = base;
  uint8_t* stages = base + kPBytes;
  auto score_slot = [&](int s) -> uint8_t* {
    return s < kStages ? stages + s * kStageBytes : p_tile + (s - kStages) * kStageBytes;
  };
  volatile int* abort = &bars->abort;

  const int c = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    if (kPool && ps.started) atomicAdd(ps.started, 1u);
    for (int s = 0; s < kSSlots; ++s) {
      mbar_init(&bars->full[s], kPool ? kLoaderThreads : 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&bars->vfull[s], kPool ? kLoaderThreads : 1);
      mbar_init(&bars->vempty[s], 1);
    }
    mbar_init(&bars->s_half, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_hi, kSoftmaxThreads);
    mbar_init(&bars->p_lo, kSoftmaxThreads);
    mbar_init(&bars->o_half, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->issued = 0;
    mbar_fence_init();
    // the first score loads go out now, while the CTA still sets itself up
    // (the barriers are initialised; nobody reads the slots before waiting)
    if (!kPool) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    for (int it = 0; !kPool && it < kSSlots && it < kScoreLoads; ++it) {
      uint8_t* st = score_slot(it);
      const int kb = it % kKB, nh = it / kKB;
      mbar_expect_tx(&bars->full[it], kStageBytes);
      tma_load_3d(st, &tm_q, &bars->full[it], kb * 64, hg * kHeads, b);
      tma_load_3d(st + kQBytes, &tm_k, &bars->full[it], kb * 64, c * kChunk + nh * kHalfRows, b);
      bars->issued = it + 1;
    }
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (kPool && (warp == 0 || warp >= 10)) {
    // ---------------- loaders: rows straight from the pool ----------------
    // The chunk's 512 pool rows first (relative to the request, into shared
    // memory); then per stage every loader thread copies its 16-byte pieces
    // into the tile's 128-byte-swizzled layout (a piece c of a stage is row
    // c >> 3, 16-byte column c & 7; 8 consecutive threads read one 128-byte
    // run). Each thread's arrival on the stage's barrier (count: all 128
    // loaders) comes from the hardware once its copies have landed; the MMA
    // thread then makes them visible to the tensor cores' async proxy. Positions
    // past k read row k-1 (their weights are zero); heads past H read head
    // H-1 (their outputs are not stored).
    const int lt = warp == 0 ? lane : (warp - 9) * 32 + lane;  // 0..255
    const int M = min(max(__ldg(ps.miss_count + b), 0), k);
    const bool repeats = __ldg(ps.miss_rows + b) != __ldg(ps.miss_count + b);
    const int j0 = c * kChunk;
    int bad = 0;
    for (int p = lt; p < kChunk; p += kLoaderThreads)
      ridx[p] = static_cast<uint16_t>(pool_row(ps, b, k, min(j0 + p, k - 1), M, repeats, bad));
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (bad && lane == 0) report(err, bad);
    // streamed: the request's staged rows of this layer are all stored (the
    // other loaders' copies follow the barrier, which orders them after this
    // thread's acquire)
    if (ps.arrived && lt == 0 &&
        !wait_word_geq(ps.arrived + b, static_cast<uint32_t>(M), ps.gather_failed, wait_ns)) {
      report(err, TS_DEVERR_TIMEOUT);
      *abort = 1;
    }
    loader_sync();
    const uint8_t* prow0 = ps.rows + int64_t(b) * ps.prow * DSA_ROW_BYTES;
    auto row_src = [&](int p) { return prow0 + int64_t(ridx[p]) * DSA_ROW_BYTES; };
    // a stage's barrier gets this thread's arrival from the hardware once its
    // copies so far have landed; the thread does not wait for them
    auto issued_stage = [&](uint64_t* bar) {
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                   : "memory");
    };
    bool ok = *abort == 0;
    for (int it = 0; it < kScoreLoads && ok; ++it) {
      const int s = it % kSSlots;
      if (it >= kSSlots) ok = warp_wait(&bars->empty[s], ((it / kSSlots) - 1) & 1, abort, wait_ns);
      if (!ok) break;
      const int kb = it % kKB, nh = it / kKB;
      uint8_t* st = score_slot(s);
#pragma unroll
      for (int i = 0; i < kHeads * 8 / kLoaderThreads; ++i) {
        const int pc = lt + kLoaderThreads * i, h = pc >> 3, col = pc & 7;
        const int hh = min(hg * kHeads + h, H - 1);
        cp_async16(st + h * 128 + ((col ^ (h & 7)) << 4),
                   ps.q + (int64_t(b) * H + hh) * DSA_ROW_BYTES + kb * 128 + col * 16);
      }
#pragma unroll
      for (int i = 0; i < kHalfRows * 8 / kLoaderThreads; ++i) {
        const int pc = lt + kLoaderThreads * i, r = pc >> 3, col = pc & 7;
        cp_async16(st + kQBytes + r * 128 + ((col ^ (r & 7)) << 4),
                   row_src(nh * kHalfRows + r) + kb * 128 + col * 16);
      }
      issued_stage(&bars->full[s]);
    }
    // value phase, once the scores are done (their slots are free then):
    // piece c of a stage is row c >> 5 of the 64-row block, dim box
    // (c >> 3) & 3, 16-byte column c & 7
    if (ok) ok = warp_wait(&bars->s_full, 0, abort, wait_ns);
    for (int v = 0; v < kLoads - kScoreLoads && ok; ++v) {
      const int s = v % kVSlots;
      if (v >= kVSlots) ok = warp_wait(&bars->vempty[s], ((v / kVSlots) - 1) & 1, abort, wait_ns);
      if (!ok) break;
      const int half = v >> 3, rb = ((v & 7) + 4) & 7;
      uint8_t* st = stages + s * kVBytes;
#pragma unroll
      for (int i = 0; i < 64 * 32 / kLoaderThreads; ++i) {
        const int pc = lt + kLoaderThreads * i, r = pc >> 5, j = (pc >> 3) & 3, col = pc & 7;
        cp_async16(st + j * kVBox + r * 128 + ((col ^ (r & 7)) << 4),
                   row_src(rb * 64 + r) + (half * 256 + j * 64) * 2 + col * 16);
      }
      issued_stage(&bars->vfull[s]);
    }
    cp_async_wait<0>();  // every copy landed before the CTA may leave
  } else if (!kPool && warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // score phase: kSSlots slots; slots 2 and 3 borrow the P region, which
      // the softmax fills only after every score product has completed (the
      // first kSSlots loads were issued during the setup)
      for (int it = bars->issued; it < kScoreLoads; ++it) {
        const int s = it % kSSlots;
        if (it >= kSSlots &&
            !mbar_wait_bounded(&bars->empty[s], ((it / kSSlots) - 1) & 1, abort, wait_ns))
          break;
        uint8_t* st = score_slot(s);
        const int kb = it % kKB, nh = it / kKB;
        mbar_expect_tx(&bars->full[s], kStageBytes);
        tma_load_3d(st, &tm_q, &bars->full[s], kb * 64, hg * kHeads, b);
        tma_load_3d(st + kQBytes, &tm_k, &bars->full[s], kb * 64, c * kChunk + nh * kHalfRows, b);
        bars->issued = it + 1;
      }
      // value phase: kVSlots slots in the ring region, once the scores are
      // done (their slots are free then); the first loads overlap the softmax
      if (bars->issued == kScoreLoads &&
          mbar_wait_bounded(&bars->s_full, 0, abort, wait_ns)) {
        for (int v = 0; v < kLoads - kScoreLoads; ++v) {
          const int s = v % kVSlots;
          if (v >= kVSlots &&
              !mbar_wait_bounded(&bars->vempty[s], ((v / kVSlots) - 1) & 1, abort, wait_ns))
            break;
          uint8_t* st = stages + s * kVBytes;
          const int half = v >> 3, rb = ((v & 7) + 4) & 7;
          mbar_expect_tx(&bars->vfull[s], kVBytes);
          for (int j = 0; j < 4; ++j)
            tma_load_3d(st + j * kVBox, &tm_v, &bars->vfull[s], half * 256 + j * 64,
                        c * kChunk + rb * 64, b);
          bars->issued = kScoreLoads + v + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(kHeads, kHalfRows, false, false);
      const uint32_t id_pv = idesc_bf16_f32(kHeads, 256, false, true);
      bool ok = true;
      for (int it = 0; it < kScoreLoads && ok; ++it) {
        const int s = it % kSSlots;
        ok = mbar_wait_bounded(&bars->full[s], (it / kSSlots) & 1, abort, wait_ns);
        if (!ok) break;
        if (kPool) fence_proxy_async_smem();  // copies written by the loaders' cp.async
        tc_fence_after();
        const int kb = it % kKB, nh = it / kKB;
        const uint32_t qa = smem_addr(score_slot(s));
        const uint32_t ka = qa + kQBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem + nh * kHalfRows, smem_desc_sw128(qa + kk * 32, 16, 1024),
                      smem_desc_sw128(ka + kk * 32, 16, 1024), id_s, (kb | kk) != 0);
        tc_commit(&bars->empty[s]);
        if (it == kKB - 1) tc_commit(&bars->s_half);
      }
      if (ok) tc_commit(&bars->s_full);
      // value products: row blocks 4..7 first, as soon as their weights are
      // written (the softmax reads the S columns they overwrite first), then
      // 0..3; dims 0..255 go to TMEM columns 256..511, dims 256..511 to
      // columns 0..255 once every S column has been read
      for (int v = 0; v < kLoads - kScoreLoads && ok; ++v) {
        const int s = v % kVSlots;
        if (v == 0 || v == 4) {
          ok = mbar_wait_bounded(v == 0 ? &bars->p_hi : &bars->p_lo, 0, abort, wait_ns);
          if (!ok) break;
        }
        ok = mbar_wait_bounded(&bars->vfull[s], (v / kVSlots) & 1, abort, wait_ns);
        if (!ok) break;
        if (kPool) fence_proxy_async_smem();
        tc_fence_after();
        const int half = v >> 3, rb = ((v & 7) + 4) & 7;
        const uint32_t d = tmem + (half == 0 ? 256u : 0u);
        const uint32_t pa = smem_addr(p_tile) + rb * kPBlock;
        const uint32_t va = smem_addr(stages + s * kVBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(d, smem_desc_sw128(pa + kk * 32, 16, 1024),
                      smem_desc_sw128(va + kk * 2048, kVBox, 1024), id_pv,
                      ((v & 7) | kk) != 0);
        tc_commit(&bars->vempty[s]);
        if (v == 7) tc_commit(&bars->o_half);
      }
      if (ok) tc_commit(&bars->o_full);
    }
  } else if (warp < 10) {
    // ---------------- softmax and epilogue: two threads per head ----------------
    // Every softmax_sync below is reached by all 256 softmax threads whatever
    // happened before it (a wait that gave up only skips work).
    const int q4 = warp & 3;            // TMEM lane quarter this warp may access
    const int part = (warp - 2) >> 2;   // which half of the chunk's columns
    const int row = q4 * 32 + lane;     // head within the tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int nvalid = min(kChunk, k - c * kChunk);
    float m = -INFINITY, l = 0.f;
    // Row max in two passes of 128 columns per thread: the first 256 rows'
    // scores are read while the tensor core computes the other 256.
    bool ok = true;
    for (int h = 0; h < 2 && ok; ++h) {
      ok = warp_wait(h == 0 ? &bars->s_half : &bars->s_full, 0, abort, wait_ns);
      if (!ok) break;
      tc_fence_after();
      const int cm = h * kHalfRows + part * (kHalfRows / 2);
      uint32_t r[32], r2[32];
      for (int cb = 0; cb < kHalfRows / 2; cb += 64) {
        tmem_ld32(trow + cm + cb, r);
        tmem_ld32(trow + cm + cb + 32, r2);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (cm + cb + i < nvalid) m = fmaxf(m, __uint_as_float(r[i]) * scale_log2);
          if (cm + cb + 32 + i < nvalid) m = fmaxf(m, __uint_as_float(r2[i]) * scale_log2);
        }
      }
    }
    if (ok) {
      if (part == 1) bars->red[row] = m;
    }
    // the row max: part 1 hands its half over, part 0 combines and hands the
    // result back (finite: column 0 is valid)
    softmax_sync();
    if (ok && part == 0) {
      m = fmaxf(m, bars->red[row]);
      bars->red[row] = m;
    }
    softmax_sync();
    if (ok) {
      if (part == 1) m = bars->red[row];
      uint32_t r[32];
      // columns 256..511 first (their P blocks feed the first value
      // products, and O's first half takes their TMEM columns), then 0..255
      for (int ph = 0; ph < 2; ++ph) {
      const int col0 = (ph == 0 ? kHalfRows : 0) + part * (kHalfRows / 2);
      for (int cb = 0; cb < kHalfRows / 2; cb += 32) {
        tmem_ld32(trow + col0 + cb, r);
        tmem_wait_ld();
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c0 = col0 + cb + 2 * i;
          const float p0 =
              c0 < nvalid ? fast_exp2(__uint_as_float(r[2 * i]) * scale_log2 - m) : 0.f;
          const float p1 =
              c0 + 1 < nvalid ? fast_exp2(__uint_as_float(r[2 * i + 1]) * scale_log2 - m) : 0.f;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          l += __low2float(h2) + __high2float(h2);
          packed[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        const int cc = col0 + cb;  // first of these 32 columns
        uint8_t* blk = p_tile + (cc >> 6) * kPBlock + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = ((cc & 63) >> 3) + j;
          *reinterpret_cast<uint4*>(blk + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ph == 0 ? &bars->p_hi : &bars->p_lo);
      }
    }
    softmax_sync();  // part 1 has read the max
    if (ok && part == 1) bars->red[row] = l;
    softmax_sync();
    if (ok && part == 0) l += bars->red[row];  // the row sum (only part 0 holds it)
    if (ok) ok = warp_wait(&bars->o_half, 0, abort, wait_ns);
    // Epilogue: O straight from TMEM to the workspace, in the chunk's
    // dim-major tile [512 dims][128 heads]: a warp's 32 lanes are 32
    // consecutive heads, so every store is a coalesced 128-byte run. Dims
    // 0..255 (TMEM columns 256..511) go out while the tensor core still
    // computes dims 256..511 (columns 0..255).
    const size_t slot0 = ((size_t(b) * HG + hg) * C + c) * kHeads;
    const int rows_valid = min(kHeads, H - hg * kHeads);
    float* tile = opart + slot0 * DSA_DV;
    bool live = ok && !*abort;
    for (int half = 0; half < 2 && live; ++half) {
      if (half == 1) {
        live = warp_wait(&bars->o_full, 0, abort, wait_ns) && !*abort;
        if (!live) break;
      }
      tc_fence_after();
      uint32_t r[32];
      for (int qq = 0; qq < 4; ++qq) {
        const int d = 128 * part + 32 * qq;  // dim within this half
        tmem_ld32(trow + (half == 0 ? 256u + d : uint32_t(d)), r);
        tmem_wait_ld();
        if (row < rows_valid) {
          float* dst = tile + size_t(256 * half + d) * kHeads + row;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i * kHeads] = __uint_as_float(r[i]);
        }
      }
    }
    if (live && part == 0 && row < rows_valid) ml[slot0 + row] = make_float2(m, l);
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    if (threadIdx.x == 0) report(err, TS_DEVERR_TIMEOUT);
    if (!kPool && warp == 0 && lane == 0) {
      // let the copies already issued land before the CTA exits: the last
      // load of every slot (earlier ones completed before their slot's reuse)
      const int issued = bars->issued;
      for (int it = issued - kSSlots < 0 ? 0 : issued - kSSlots; it < issued; ++it) {
        if (it < kScoreLoads) {
          mbar_wait_timed(&bars->full[it % kSSlots], (it / kSSlots) & 1, kWaitLimit);
        } else {
          const int v = it - kScoreLoads;
          mbar_wait_timed(&bars->vfull[v % kVSlots], (v / kVSlots) & 1, kWaitLimit);
        }
      }
    }
    if (warp == 1 && lane == 0) {
      // every tcgen05 operation this thread issued completes before the free
      tc_commit(&bars->drain);
      mbar_wait_timed(&bars->drain, 0, kWaitLimit);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the chunks of a (request, head tile), kCombineDims dims per CTA, one thread per
// head: out = sum_c w_c O_c / sum_c w_c l_c with w_c = exp2(m_c - max_c m_c).
// The chunks' tiles are dim-major, so each load of a warp is one coalesced
// 128-byte run; the result goes out through shared memory as 16-byte row
// pieces.
constexpr int kCombineDims = 16;
__global__ void __launch_bounds__(kHeads) sfa_combine_kernel(const float* __restrict__ opart,
                                                             const float2* __restrict__ ml, int H,
                                                             int HG, int C,
                                                             __nv_bfloat16* __restrict__ out,
                                                             float* __restrict__ lse) {
  __shared__ __align__(16) __nv_bfloat16 tile[kHeads][kCombineDims + 8];
  const int db = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int h = threadIdx.x;
  const int rows_valid = min(kHeads, H - hg * kHeads);
  const size_t s0 = ((size_t(b) * HG + hg) * C) * kHeads;  // chunk 0, head 0
  if (h < rows_valid) {
    float mx = -INFINITY;
    for (int c = 0; c < C; ++c) mx = fmaxf(mx, __ldg(ml + s0 + size_t(c) * kHeads + h).x);
    float denom = 0.f;
    float acc[kCombineDims];
#pragma unroll
    for (int i = 0; i < kCombineDims; ++i) acc[i] = 0.f;
    for (int c = 0; c < C; ++c) {
      const float2 e = __ldg(ml + s0 + size_t(c) * kHeads + h);
      const float w = exp2f(e.x - mx);
      denom += w * e.y;
      const float* src = opart + (s0 + size_t(c) * kHeads) * DSA_DV +
                         size_t(db) * kCombineDims * kHeads + h;
#pragma unroll
      for (int i = 0; i < kCombineDims; ++i) acc[i] += w * __ldcs(src + i * kHeads);
    }
    const float inv = 1.f / denom;
#pragma unroll
    for (int i = 0; i < kCombineDims; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(&tile[h][i]) =
          __floats2bfloat162_rn(acc[i] * inv, acc[i + 1] * inv);
    if (db == 0 && lse) lse[size_t(b) * H + hg * kHeads + h] = mx * kLn2 + logf(denom);
  }
  __syncthreads();
  // rows_valid rows of kCombineDims dims, in 16-byte pieces
  constexpr int kPieces = kCombineDims / 8;
  for (int j = h; j < kHeads * kPieces; j += kHeads) {
    const int r = j / kPieces, piece = j - r * kPieces;
    if (r < rows_valid)
      *reinterpret_cast<uint4*>(out + (size_t(b) * H + hg * kHeads + r) * DSA_DV +
                                db * kCombineDims + piece * 8) =
          *reinterpret_cast<const uint4*>(&tile[r][piece * 8]);
  }
}

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// 3-D map over rows of 576 bf16: dims {576, rows, batch}; box {64, box_rows, 1}.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t batch, uint32_t box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {DSA_D, rows, batch};
  const cuuint64_t strides[2] = {DSA_ROW_BYTES, rows * DSA_ROW_BYTES};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The attention's two launches, from a selection buffer (sel_l; ps unused) or
// straight from a staged-layout pool (kPool: ps): the chunks, then their merge.
template <bool kPool>
ts_status launch_attention(const void* q, const void* rows, const PoolSrc& ps, int B, int H,
                           int k, float scale, void* out, float* lse, void* ws, int32_t* err,
                           cudaStream_t stream) {
  const int HG = (H + kHeads - 1) / kHeads, C = (k + kChunk - 1) / kChunk;
  // the tile variant loads through tensor maps; the pool variant's loader
  // warps copy with plain addresses (its maps stay unused)
  CUtensorMap tm_q = {}, tm_k = {}, tm_v = {};
  if (!kPool && (!make_map(&tm_q, q, H, B, kHeads) || !make_map(&tm_k, rows, k, B, kHalfRows) ||
                 !make_map(&tm_v, rows, k, B, 64)))
    return TS_ERR_CUDA;
  const uint32_t smem = kPool ? kPoolSmemBytes : kSmemBytes;
  const int threads = kPool ? kPoolThreads : kThreads;
  const size_t slots = size_t(B) * HG * C * kHeads;
  float* opart = static_cast<float*>(ws);
  float2* ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + align256(slots * DSA_DV * 4));
  static std::atomic<uint64_t> smem_set{0};
  if (!raise_smem_limit(reinterpret_cast<const void*>(sfa_chunk_kernel<kPool>),
                        static_cast<int>(smem), smem_set))
    return TS_ERR_CUDA;
  sfa_chunk_kernel<kPool><<<dim3(C, HG, B), threads, smem, stream>>>(
      tm_q, tm_k, tm_v, H, k, HG, C, scale * kLog2e, opart, ml, wait_limit_ns(kWaitLimit), ps,
      err);
  if (launch_status() != TS_OK) return TS_ERR_CUDA;
  sfa_combine_kernel<<<dim3(DSA_DV / kCombineDims, HG, B), kHeads, 0, stream>>>(
      opart, ml, H, HG, C, static_cast<__nv_bfloat16*>(out), lse);
  return launch_status();
}

}  // namespace
}  // namespace dsakv

using namespace dsakv;

extern "C" size_t sfa_workspace_size(int B, int H, int k) {
  if (B <= 0 || H <= 0 || k <= 0) return 0;
  const size_t HG = (H + kHeads - 1) / kHeads, C = (k + kChunk - 1) / kChunk;
  const size_t slots = size_t(B) * HG * C * kHeads;
  return align256(slots * DSA_DV * 4) + align256(slots * 8);
}

namespace dsakv {

ts_status sfa_check(const void* q, const void* sel_l, int B, int H, int k, float scale,
                    void* out, const void* ws, size_t ws_bytes) {
  if (!q || !sel_l || !out || !ws) return TS_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || k <= 0 || !std::isfinite(scale)) return TS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(sel_l) || !aligned16(out)) return TS_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535 * kHeads || int64_t(B) * H > 2147483647) return TS_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < sfa_workspace_size(B, H, k))
    return TS_ERR_WORKSPACE;
  return TS_OK;
}

uint32_t sfa_chunk_ctas(int B, int H, int k) {
  return uint32_t((k + kChunk - 1) / kChunk) * uint32_t((H + kHeads - 1) / kHeads) * uint32_t(B);
}

ts_status sfa_enqueue(const void* q, const void* sel_l, int B, int H, int k, float scale,
                      void* out, float* lse, void* ws, int32_t* err, cudaStream_t stream) {
  return launch_attention<false>(q, sel_l, PoolSrc{}, B, H, k, scale, out, lse, ws, err, stream);
}

ts_status sfa_pool_check(const void* q, const void* pool_l, int P, const int32_t* src_map,
                         const int32_t* miss_ids, const int32_t* miss_pos,
                         const int32_t* miss_count, const int32_t* miss_rows, int B, int H, int k,
                         float scale, void* out, const void* ws, size_t ws_bytes) {
  const ts_status st = sfa_check(q, pool_l, B, H, k, scale, out, ws, ws_bytes);
  if (st != TS_OK) return st;
  if (!src_map || !miss_ids || !miss_pos || !miss_count || !miss_rows || P <= 0)
    return TS_ERR_INVALID_ARG;
  if (int64_t(B) * (int64_t(P) + k) >= (int64_t(1) << 31) || int64_t(P) + k > 65536)
    return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

ts_status sfa_pool_enqueue(const void* q, const void* pool_l, int P, const int32_t* src_map,
                           const int32_t* miss_ids, const int32_t* miss_pos,
                           const int32_t* miss_count, const int32_t* miss_rows, int B, int H,
                           int k, float scale, void* out, float* lse, void* ws, int32_t* err,
                           cudaStream_t stream, const uint32_t* arrived,
                           const uint32_t* gather_failed, uint32_t* started) {
  if (arrived && !gather_failed) return TS_ERR_INVALID_ARG;
  const PoolSrc ps{src_map, miss_ids, miss_pos, miss_count, miss_rows,
                   static_cast<const uint8_t*>(pool_l), static_cast<const uint8_t*>(q), P, P + k,
                   arrived, gather_failed, started};
  return launch_attention<true>(q, pool_l, ps, B, H, k, scale, out, lse, ws, err, stream);
}

}  // namespace dsakv

extern "C" ts_status sfa_mla_decode(const void* q, const void* sel_l, int B, int H, int k,
                                    float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                    int32_t* err, cudaStream_t stream) {
  const ts_status st = sfa_check(q, sel_l, B, H, k, scale, out, ws, ws_bytes);
  if (st != TS_OK) return st;
  return sfa_enqueue(q, sel_l, B, H, k, scale, out, lse, ws, err, stream);
}

extern "C" ts_status sfa_mla_decode_pool(const void* q, const void* pool_l, int P,
                                         const int32_t* src_map, const int32_t* miss_ids,
                                         const int32_t* miss_pos, const int32_t* miss_count,
                                         const int32_t* miss_rows, int B, int H, int k,
                                         float scale, void* out, float* lse, void* ws,
                                         size_t ws_bytes, int32_t* err, cudaStream_t stream) {
  const ts_status st = sfa_pool_check(q, pool_l, P, src_map, miss_ids, miss_pos, miss_count,
                                      miss_rows, B, H, k, scale, out, ws, ws_bytes);
  if (st != TS_OK) return st;
  return sfa_pool_enqueue(q, pool_l, P, src_map, miss_ids, miss_pos, miss_count, miss_rows, B, H,
                          k, scale, out, lse, ws, err, stream);
}
