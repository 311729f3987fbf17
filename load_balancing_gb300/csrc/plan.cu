// LPT planning with a stay-in-place bonus, on the device, bit-exact.
//
// db-SP blog, scenario 1: the longest remaining item goes to the least-loaded
// worker (LPT, the greedy for identical-machines scheduling). db-SP blog,
// scenario 2, third bullet: an item placed on its original worker counts as
// lighter when the worker is chosen. Readings: equal loads are taken by ascending
// id, ties between workers go to the lowest index, the bonus enters only the
// choice and the worker accrues the item's true load.
//
// Worker keys are packed as (load << 11 | worker), so the greedy's choice (lowest
// load, then lowest index) is the smallest key: 32-bit when every worker load stays
// below 2^20 (LPT keeps the largest below total / m + max_load), else 64-bit. One
// CTA of 256 threads:
//
//   phase 0  check loads and home, find the load range; when n <= 45056 and every
//            load <= 2047 the loads are staged in shared memory as uint16
//            ("staged" path), otherwise the kernel works from global memory;
//   phase 1  the stable order (load desc, id asc): a counting sort through
//            shared-memory histograms, its stable scatter done per warp with match_any
//            (groups of ids of one load at once; one warp over the worklist when the
//            loads are not staged, rank-by-comparison for n <= 16384 with large loads);
//   phase 2  the greedy.
//            Without a bonus (whole CTA) it goes in batches over the workers' keys sorted
//            ascending in A: the next items take A[0], A[1], ... while A[j] stays below
//            A[0] + W(s + j), exactly the one-at-a-time greedy's picks (every warp finds
//            the end of the batch by ballots, without a block barrier), then A is rebuilt
//            by a counting sort over a ring of load buckets (when the loads are staged
//            and small), else the re-keyed keys are merged back by binary searches.
//            With a bonus (one warp) the key of item i's home worker is lowered by the
//            bonus for that choice only, so items go one at a time: every lane keeps the
//            keys of workers lane, lane+32, ... in registers and one warp minimum (two
//            for 64-bit keys) decides an item. A bonus above the total load keeps every
//            item at home: one warp ranks each worker's items in the stable order.
//            worker_of[i] temporarily holds worker + cm * (rank within worker), cm = 1024
//            (or m when ranks could reach 2^21);
//   phase 3  CSR offsets by a block scan of the per-worker counts, then the
//            scatter of every item to offsets[worker] + rank.
// Phases 0, 1 and 3 keep 8 global reads in flight per thread from 16,384 items up and 4
// below; a launch runs one of the two instantiations. Global working storage is the
// output arrays only.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kStagedMaxItems = 45056;
constexpr int kStagedMaxLoad = 2047;
constexpr int kMaxLoadCounting = 32767;
constexpr int kMaxItemsCompare = 16384;
constexpr int kWorkerBits = 11;  // worker index < 2048 in the packed key
constexpr long long kWorkerMask = (1LL << kWorkerBits) - 1;
constexpr long long kKeyNone = LLONG_MAX;
constexpr int kRunLoadBits = 11;  // runs of equal load: (end << 11 | load), load <= kStagedMaxLoad
constexpr int kRunLoadMask = (1 << kRunLoadBits) - 1;
static_assert(kStagedMaxLoad <= kRunLoadMask && (long long)kStagedMaxItems << kRunLoadBits < (1LL << 31),
              "a run's end and load share one int");
static_assert(2 * DBSP_MAX_WORKERS * 2 >= kStagedMaxLoad + 1, "the run table fits the key array");

constexpr size_t kStagedBytes = 2ull * kStagedMaxItems + 4ull * (kStagedMaxLoad + 2) + 4ull * 8 * (kStagedMaxLoad + 1);
constexpr size_t kGlobalBytes = 4ull * (kMaxLoadCounting + 2 > kMaxItemsCompare ? kMaxLoadCounting + 2 : kMaxItemsCompare);
constexpr size_t kDynBytes0 = kStagedBytes > kGlobalBytes ? kStagedBytes : kGlobalBytes;

struct PlanShared {
  int min_load, max_load, bad_home;
  unsigned long long total_load;
  int scan[kThreads / 32 + 1];
};

// offset of the bucket ring in the dynamic buffer: past the staged order and its cursor
constexpr size_t kRingOff = (2ull * kStagedMaxItems + 4ull * (kStagedMaxLoad + 2) + 15) / 16 * 16;
constexpr int kRingWordsMax = 10240;  // bucket words R * ceil(m / 32)
constexpr int kRingMax = 4096;        // buckets R
constexpr size_t kPreOff = kRingOff + 4ull * kRingWordsMax;   // scan of the bucket counts
constexpr size_t kCntOff = kPreOff + 4ull * kRingMax;         // bucket counts
constexpr size_t kLwOff = kCntOff + 4ull * kRingMax;          // stored load of each worker
constexpr size_t kAOff = kLwOff + 4ull * DBSP_MAX_WORKERS;    // sorted keys
constexpr size_t kRingEnd = kAOff + 8ull * DBSP_MAX_WORKERS;
constexpr size_t kDynBytes = kDynBytes0 > kRingEnd ? kDynBytes0 : kRingEnd;

// Global reads in flight per thread in phases 0, 1 and 3, as a type: 8 from kDeepItems
// items up, 4 below. Both depths are instantiated and a launch runs one, so a small plan
// fetches (cold) only the shorter code.
template <int U>
struct Depth {
  static constexpr int value = U;
};
constexpr int kDeepItems = 16384;

// Exclusive scan over `n` ints in shared memory `a` (in place). All threads call it.
__device__ void block_exclusive_scan(int* a, int n, int* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int s = 0;
  for (int j = lo; j < hi; ++j) s += a[j];
  int x = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < kThreads / 32; ++w) { const int t = warp_sums[w]; warp_sums[w] = run; run += t; }
  }
  __syncthreads();
  int run = warp_sums[warp] + x - s;
  for (int j = lo; j < hi; ++j) { const int t = a[j]; a[j] = run; run += t; }
  __syncthreads();
}

template <int KMAX>
__device__ __forceinline__ long long lane_minimum(const long long (&key)[KMAX]) {
  long long m = key[0];
#pragma unroll
  for (int q = 1; q < KMAX; ++q) m = key[q] < m ? key[q] : m;
  return m;
}

struct Sorted {  // the stable order, staged in shared memory or in the worklist
  const uint16_t* smem;
  const int32_t* gmem;
  __device__ __forceinline__ int operator[](int t) const { return smem ? (int)smem[t] : gmem[t]; }
};

// Phase 2 without a bonus: batches per run of equal loads, on the whole CTA.
// The worker keys stay sorted in a circular list: logical key i is A[(h + i) mod m].
// One batch of a run with load w (wk = w << 11), b = number of keys below
// A[h] + wk:
//   * b > 1: the next bp = min(b, r) items take the first bp keys in order (each
//     re-keyed key is at or above the threshold, above every key still in the
//     batch), so the one-at-a-time greedy makes exactly these picks;
//   * b == 1: the minimum keeps winning while its key stays below the runner-up,
//     for q = ceil((key1 - key0) / wk) picks, and is re-keyed once by q * wk.
// Then the head advances past the picked keys; the keys below the threshold do not
// move, and only the "tail" (keys at or above the threshold) is merged with the
// re-keyed keys: every element is placed by a binary search in the other list, KT
// elements per thread, all searches of a batch in parallel.
template <int KT, typename K>
__device__ void greedy_batched(const Sorted sorted, const int* bin_end, int nbins, int max_load, int n, int m,
                               int cm, int bc, int ic, K* A, int* counts, long long* final_load,
                               int32_t* __restrict__ worker_of, int* red) {
  constexpr int kW = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int j = tid; j < m; j += kThreads) { A[j] = j; counts[j] = 0; }
  __syncthreads();
  int h = 0;
  auto phys = [&](int i) { const int x = h + i; return x >= m ? x - m : x; };
  int s = 0;
  for (int bin = 0; bin < nbins && s < n; ++bin) {
    const int e = bin_end[bin];
    int r = e - s;
    if (r <= 0) continue;
    const int w = (max_load - bin) * bc + ic;  // the planning load of this run's items
    if (w == 0) {  // zero loads never change a key: they all go to the current minimum
      const int p0 = (int)(A[h] & (K)kWorkerMask);
      const int base = counts[p0];
      for (int j = tid; j < r; j += kThreads) worker_of[sorted[s + j]] = p0 + cm * (base + j);
      __syncthreads();
      if (tid == 0) counts[p0] = base + r;
      __syncthreads();
      s = e;
      continue;
    }
    const K wk = (K)w << kWorkerBits;
    while (r > 0) {
      const K key0 = A[h];
      const K thr = key0 + wk;
      int c = 0;
#pragma unroll
      for (int t = 0; t < KT; ++t) {  // order does not matter for a count
        const int j = tid + kThreads * t;
        c += (j < m) && A[j < m ? j : 0] < thr;
      }
      c = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) red[warp] = c;
      __syncthreads();
      int b = 0;
#pragma unroll
      for (int q = 0; q < kW; ++q) b += red[q];
      int bp, picks, p1 = -1, base1 = 0;
      K step;  // amount added to each picked key
      if (b == 1) {
        picks = m > 1 ? (int)min((long long)r, (long long)((A[phys(1)] - key0 + wk - 1) / wk)) : r;
        bp = 1;
        step = (K)picks * wk;
        p1 = (int)(key0 & (K)kWorkerMask);
        base1 = counts[p1];
        for (int j = tid; j < picks; j += kThreads) worker_of[sorted[s + j]] = p1 + cm * (base1 + j);
      } else {
        bp = min(b, r);
        picks = bp;
        step = wk;
        for (int j = tid; j < bp; j += kThreads) {  // distinct workers: no two threads share a count
          const int p = (int)(A[phys(j)] & (K)kWorkerMask);
          const int rank = counts[p];
          counts[p] = rank + 1;
          worker_of[sorted[s + j]] = p + cm * rank;
        }
      }
      // merge region: new logical positions [b - bp, m) after the head moves by bp;
      // element k < bp is the re-keyed key Y_k = key(k) + step, element k >= bp the
      // tail key at logical b + (k - bp)
      const int E = bp + (m - b);
      const int h_new = phys(bp);
      K val[KT], add[KT];
      int lo[KT], hi[KT], depth[KT];
#pragma unroll
      for (int t = 0; t < KT; ++t) {
        const int k = tid + kThreads * t;
        const bool live = k < E;
        const bool is_y = k < bp;
        int src = is_y ? k : b + k - bp;
        src = live ? src : 0;
        const K a = A[phys(src)];
        val[t] = is_y ? a + step : a;
        add[t] = is_y ? (K)0 : step;  // a tail key is compared with re-keyed keys: add the step
        lo[t] = !live ? 0 : (is_y ? b : 0);
        hi[t] = !live ? 0 : (is_y ? m : bp);
        depth[t] = 32 - __clz(hi[t] - lo[t]);  // halvings for the list searched
      }
      int iters = 0;
#pragma unroll
      for (int t = 0; t < KT; ++t) iters = max(iters, depth[t]);
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int t = 0; t < KT; ++t) {
          const int mid = (lo[t] + hi[t]) >> 1;  // lo == hi <= m still indexes the list
          int x = h + mid;
          x = x >= m ? x - m : x;
          x = x >= m ? x - m : x;
          const K am = A[x] + add[t];
          const bool go = lo[t] < hi[t];
          const bool less = am < val[t];
          lo[t] = go && less ? mid + 1 : lo[t];
          hi[t] = go && !less ? mid : hi[t];
        }
      }
      int dst[KT];
#pragma unroll
      for (int t = 0; t < KT; ++t) {
        const int k = tid + kThreads * t;
        const int pos = k < bp ? (b - bp) + k + (lo[t] - b) : (b - bp) + (k - bp) + lo[t];
        int x = h_new + pos;
        x = x >= m ? x - m : x;
        dst[t] = k < E ? x : -1;
      }
      __syncthreads();  // every read of the old order and of the counts is done
#pragma unroll
      for (int t = 0; t < KT; ++t)
        if (dst[t] >= 0) A[dst[t]] = val[t];
      if (tid == 0 && p1 >= 0) counts[p1] = base1 + picks;
      __syncthreads();
      h = h_new;
      s += picks;
      r -= picks;
    }
  }
  for (int j = tid; j < m; j += kThreads) final_load[A[j] & (K)kWorkerMask] = (long long)(A[j] >> kWorkerBits);
}

// Phase 2 without a bonus when the planning loads are small: sorted keys, rebuilt by a
// counting sort over a ring of load buckets.
//
// A holds the workers' keys (load << 11 | worker) in ascending order. A batch takes
// the next items s, s+1, ... in the stable order: item s + j goes to worker A[j] for
// every j below bp = #{j : A[j] < A[0] + W(s + j)} (W the item's planning load, shifted
// like the keys). That is exactly the one-at-a-time greedy: A[j] - W(s + j) grows with
// j (keys ascend, loads descend), so the predicate holds for j < bp only, and when item
// s + j is placed every earlier pick already carries A[i] + W(s + i) >= A[0] + W(s + j)
// > A[j] while the later keys are larger, so A[j] is the minimum. A batch may span runs
// of different loads. Two shortcuts:
//   * bp == 1: the minimum keeps winning while its key stays below the runner-up's,
//     q = ceil((A[1] - A[0]) / W) picks within the run;
//   * bp == m with m or more items of one load left in the run: every later round of m
//     items keeps the same order, so floor(r / m) whole rounds are placed at once and
//     every load grows by the same amount (kept aside as a shift).
// The load of a sorted position is read off the staged loads (sload) where they fit beside
// the order; otherwise from a table of the runs of equal load (the non-empty load bins
// only, run[k] = (one past the run's last position << 11 | its load)), so that finding the
// run of a position never walks the empty bins between two loads (a handful of distinct
// loads spread over hundreds of bins on the imbalance workload).
// After a batch the picked workers move up in a ring of load buckets (bucket L mod R
// holds, as a bitmask, the workers whose stored load is L; R a power of two >= 2 wmax +
// 1, since every load stays within [L0, L0 + 2 wmax] of the minimum L0), and A is
// rebuilt by a counting sort: a worker's new position is the number of workers in
// lower buckets (an exclusive scan of the bucket counts from L0) plus the workers below
// it in its own bucket.
constexpr int kRingWords = kRingWordsMax;  // R * ceil(m / 32) bucket words

// WPT = ceil(m_max / 256) workers per thread for the instantiation's worker bound. Returns
// false (uniformly) when the state is found inconsistent (a batch without a pick, or
// more batches than items) instead of looping.
template <int WPT>
__device__ __forceinline__ bool greedy_sorted(const int32_t* __restrict__ loads, const uint16_t* __restrict__ sorted,
                                              const uint16_t* __restrict__ sload,
                                              const int* bin_end, int max_load, const int* run, int n, int m,
                                              int cm, int bc, int ic, int R, uint32_t* bkt, int* pre, int* bcnt,
                                              int* Lw,
                                              unsigned long long* A, int* counts, long long* final_load,
                                              int32_t* __restrict__ worker_of, int* red) {
  constexpr int kW = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (m == 1) {  // one worker takes every item, in order
    for (int t = tid; t < n; t += kThreads) worker_of[sorted[t]] = cm * t;
    long long tot = 0;
    for (int t = tid; t < n; t += kThreads) tot += (long long)__ldg(loads + sorted[t]) * bc + ic;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) reinterpret_cast<long long*>(A)[warp] = tot;
    __syncthreads();
    if (tid == 0) {
      long long sum = 0;
      for (int q = 0; q < kW; ++q) sum += reinterpret_cast<long long*>(A)[q];
      final_load[0] = sum;
      counts[0] = n;
    }
    __syncthreads();
    return true;
  }
  const int WPB = (m + 31) >> 5;
  const int rmask = R - 1;
  for (int j = tid; j < R * WPB; j += kThreads) {
    uint32_t v = 0;
    if (j < WPB) {  // bucket 0: every worker
      const int lo = j * 32;
      v = m - lo >= 32 ? 0xffffffffu : ((1u << (m - lo)) - 1u);
    }
    bkt[j] = v;
  }
  for (int j = tid; j < R; j += kThreads) bcnt[j] = j == 0 ? m : 0;
  for (int j = tid; j < m; j += kThreads) {
    Lw[j] = 0;
    counts[j] = 0;
    A[j] = (unsigned long long)j;
  }
  __syncthreads();
  int L0 = 0;           // stored load of A[0]
  long long shift = 0;  // load added to every worker by whole rounds
  int s = 0, k0 = 0;  // the next item and the run holding it
  long long batches = 0;
  const long long max_batches = (long long)n + 8;
  while (s < n) {
    if (++batches > max_batches) return false;
    int run_end, ls;  // the run holding item s: its end and load
    if (sload) {
      ls = sload[s];
      run_end = bin_end[max_load - ls];
    } else {
      while ((run[k0] >> kRunLoadBits) <= s) ++k0;  // (s < n, the last run's end)
      run_end = run[k0] >> kRunLoadBits;
      ls = run[k0] & kRunLoadMask;
    }
    const int ws = ls * bc + ic;  // planning load of item s
    const unsigned long long key0 = A[0];
    // every stored load after this batch lies in [L0, L0 + span): the largest is at most
    // the current largest plus ws (the items are in descending order of load)
    const int span = (int)min((long long)R, (long long)(A[m - 1] >> kWorkerBits) - L0 + ws + 1);
    const int p0 = (int)(key0 & kWorkerMask);
    if (ws == 0) {  // zero loads never change a key: the rest goes to the minimum
      const int c0 = counts[p0];
      for (int t = tid; t < n - s; t += kThreads) worker_of[sorted[s + t]] = p0 + cm * (c0 + t);
      __syncthreads();
      if (tid == 0) counts[p0] = c0 + (n - s);
      s = n;
      break;
    }
    // ---- bp: the positions j whose key is below A[0] + W(s + j). The predicate holds for a
    // prefix of j (A[j] - W(s + j) grows with j), so every warp finds its end by itself,
    // the last position first (a whole round) and then 32 positions per ballot, with no
    // block barrier; every warp reads the same keys and loads and gets the same bp.
    const int cap = min(m, n - s);
    auto wload = [&](int pos) {  // planning load of sorted position pos (s <= pos < n)
      if (pos < run_end) return ws;
      int l;
      if (sload) {
        l = sload[pos];
      } else {
        int k = k0 + 1;
        while ((run[k] >> kRunLoadBits) <= pos) ++k;  // (pos < n, the last run's end)
        l = run[k] & kRunLoadMask;
      }
      return l * bc + ic;
    };
    auto below = [&](int j) { return A[j] < key0 + ((unsigned long long)wload(s + j) << kWorkerBits); };
    int bp = cap;
    if (!below(cap - 1)) {
      for (int c = 0; c < cap; c += 32) {
        const int j = c + lane;
        const unsigned ok = __ballot_sync(0xffffffffu, j < cap && below(j));
        if (ok != 0xffffffffu) {
          bp = c + __ffs(~ok) - 1;
          break;
        }
      }
    }
    if (bp < 1) return false;
    if (bp == 1) {
      // ---- the minimum alone: it keeps winning while its key stays below the runner-up
      const unsigned long long W = (unsigned long long)ws << kWorkerBits;
      const int r = run_end - s;
      const int q = m == 1 ? r : (int)min((unsigned long long)r, (A[1] - key0 + W - 1) / W);
      const int c0 = counts[p0];
      for (int t = tid; t < q; t += kThreads) worker_of[sorted[s + t]] = p0 + cm * (c0 + t);
      __syncthreads();  // every thread read counts[p0], A[0] and A[1]
      if (tid == 0) {
        counts[p0] = c0 + q;
        const int Lo = Lw[p0], Ln = Lo + q * ws;
        const uint32_t bit = 1u << (p0 & 31);
        bkt[(Lo & rmask) * WPB + (p0 >> 5)] &= ~bit;
        bkt[(Ln & rmask) * WPB + (p0 >> 5)] |= bit;
        --bcnt[Lo & rmask];
        ++bcnt[Ln & rmask];
        Lw[p0] = Ln;
      }
      s += q;
    } else if (bp == m && run_end - s >= m) {
      // ---- whole rounds of equal loads: the order of A does not change
      const int F = (run_end - s) / m;
#pragma unroll
      for (int k = 0; k < WPT; ++k) {
        const int j = tid + k * kThreads;
        if (j < m) {
          const int p = (int)(A[j] & kWorkerMask);
          const int c0 = counts[p];
#pragma unroll 4  // the order reads of several rounds go out together
          for (int f = 0; f < F; ++f) worker_of[sorted[s + f * m + j]] = p + cm * (c0 + f);
          counts[p] = c0 + F;
        }
      }
      shift += (long long)F * ws;
      s += F * m;
      __syncthreads();  // A, counts and red are read again by the next batch
      continue;
    } else {
      // ---- a batch: item s + j to worker A[j] for j < bp; each moves up by W(s + j)
#pragma unroll
      for (int k = 0; k < WPT; ++k) {
        const int j = tid + k * kThreads;
        if (j < bp) {
          const int p = (int)(A[j] & kWorkerMask);
          const int c0 = counts[p];
          worker_of[sorted[s + j]] = p + cm * c0;
          counts[p] = c0 + 1;
          const int Lo = Lw[p], Ln = Lo + wload(s + j);
          const uint32_t bit = 1u << (p & 31);
          atomicAnd(&bkt[(Lo & rmask) * WPB + (p >> 5)], ~bit);
          atomicOr(&bkt[(Ln & rmask) * WPB + (p >> 5)], bit);
          atomicSub(&bcnt[Lo & rmask], 1);
          atomicAdd(&bcnt[Ln & rmask], 1);
          Lw[p] = Ln;
        }
      }
      s += bp;
    }
    __syncthreads();  // the buckets are final for this batch
    // ---- counting sort: exclusive scan of the bucket counts from L0 over the span
    {
      // each thread scans a slice of at most kRingMax / kThreads buckets: its counts are
      // read as independent predicated loads into registers (a short and a long form)
      const int per = (span + kThreads - 1) / kThreads;
      const int i0 = min(span, tid * per), cnt = min(span, i0 + per) - i0;
      auto scan_slice = [&](auto depth) {
        constexpr int kN = decltype(depth)::value;
        int c[kN];
        int tot = 0;
#pragma unroll
        for (int u = 0; u < kN; ++u) {
          c[u] = u < cnt ? bcnt[(L0 + i0 + u) & rmask] : 0;
          tot += c[u];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) red[warp] = incl;
        __syncthreads();
        int run = incl - tot;
#pragma unroll
        for (int q = 0; q < kW; ++q) run += q < warp ? red[q] : 0;
#pragma unroll
        for (int u = 0; u < kN; ++u) {
          if (u < cnt) pre[i0 + u] = run;
          run += c[u];
        }
      };
      static_assert(kRingMax / kThreads <= 16, "a thread's slice of the ring fits the long form");
      if (per <= 2)
        scan_slice(Depth<2>{});
      else
        scan_slice(Depth<16>{});
    }
    __syncthreads();
    int bad = 0;  // a load outside [L0, L0 + span) or a position outside [0, m): inconsistent state
#pragma unroll
    for (int k = 0; k < WPT; ++k) {
      const int p = tid + k * kThreads;
      if (p < m) {
        const int L = Lw[p];
        if ((unsigned)(L - L0) >= (unsigned)span) {
          bad = 1;
          continue;
        }
        const uint32_t* wd = bkt + (L & rmask) * WPB;
        int pos = pre[L - L0];
#pragma unroll  // the words below p's word, as independent predicated reads
        for (int q = 0; q < WPT * kThreads / 32 - 1; ++q)
          if (q < (p >> 5)) pos += __popc(wd[q]);
        pos += __popc(wd[p >> 5] & ((1u << (p & 31)) - 1u));
        if ((unsigned)pos >= (unsigned)m) {
          bad = 1;
          continue;
        }
        A[pos] = ((unsigned long long)L << kWorkerBits) | (unsigned long long)p;
      }
    }
    if (__syncthreads_or(bad)) return false;
    L0 = (int)(A[0] >> kWorkerBits);
  }
  __syncthreads();
  for (int j = tid; j < m; j += kThreads) final_load[j] = (long long)Lw[j] + shift;
  return true;
}

// Phase 2 with a bonus: one item at a time (one warp). K is int when every key fits 31
// bits (then one warp minimum per item), else long long (two, over the halves).
template <int KMAX, typename K>
__device__ __forceinline__ void greedy_serial(const Sorted sorted, const int32_t* __restrict__ loads,
                              const int32_t* __restrict__ home, int bonus, int bc, int ic, int n, int m, int cm,
                              int* counts,
                              long long* final_load, int32_t* __restrict__ worker_of) {
  constexpr K kNone = sizeof(K) == 4 ? (K)INT_MAX : (K)kKeyNone;
  const int lane = threadIdx.x & 31;
  K key[KMAX];
  int cnt[KMAX];
#pragma unroll
  for (int q = 0; q < KMAX; ++q) {
    const int p = lane + 32 * q;
    key[q] = p < m ? (K)p : kNone;  // load 0, worker p
    cnt[q] = 0;
  }
  // the lane's smallest key, as a balanced tree of minimums (log2 KMAX deep)
  auto lane_min = [&]() {
    K a[KMAX];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) a[q] = key[q];
#pragma unroll
    for (int step = 1; step < KMAX; step <<= 1) {
#pragma unroll
      for (int q = 0; q + step < KMAX; q += 2 * step) a[q] = a[q + step] < a[q] ? a[q + step] : a[q];
    }
    return a[0];
  };
  // key[idx] picked by the bits of idx, a balanced tree of selects (log2 KMAX deep)
  auto pick = [&](int idx) {
    K a[KMAX];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) a[q] = key[q];
#pragma unroll
    for (int step = 1; step < KMAX; step <<= 1) {
#pragma unroll
      for (int q = 0; q + step < KMAX; q += 2 * step) a[q] = (idx & step) ? a[q + step] : a[q];
    }
    return a[0];
  };
  K my_min = lane_min();
  const K bonus_key = (K)bonus << kWorkerBits;
  for (int base = 0; base < n; base += 32) {
    const int t = base + lane;
    int my_i = 0, my_w = 0, my_h = -1;
    if (t < n) {
      my_i = sorted[t];
      my_w = loads[my_i] * bc + ic;
      if (home) my_h = home[my_i];
    }
    const int chunk = min(32, n - base);
#pragma unroll 2  // the next item's shuffles overlap this item's chain (4 and 8 were slower)
    for (int s = 0; s < chunk; ++s) {
      const int i = __shfl_sync(0xffffffffu, my_i, s);
      const int w = __shfl_sync(0xffffffffu, my_w, s);
      const int h = __shfl_sync(0xffffffffu, my_h, s);
      // the lane holding the home worker offers its key lowered by the bonus (branch-free:
      // every lane evaluates it, so the warp never diverges on the way to the minimum)
      K kh = pick(h >> 5);  // (h >> 5 < KMAX for every worker; for h < 0 the value is unused)
      kh -= bonus_key;
      const K cand = (h >= 0 && (h & 31) == lane && kh < my_min) ? kh : my_min;
      int p;
      if constexpr (sizeof(K) == 4) {
        p = __reduce_min_sync(0xffffffffu, (int)cand) & (int)kWorkerMask;
      } else {
        const int hi = (int)(cand >> 32);
        const int min_hi = __reduce_min_sync(0xffffffffu, hi);
        const unsigned lo = hi == min_hi ? (unsigned)(cand & 0xffffffffu) : 0xffffffffu;
        const unsigned min_lo = __reduce_min_sync(0xffffffffu, lo);
        p = (int)(min_lo & (unsigned)kWorkerMask);
      }
      const bool mine = (p & 31) == lane;  // the lane holding the chosen worker
      const int qp = mine ? p >> 5 : -1;
      int rank = 0;
#pragma unroll
      for (int q = 0; q < KMAX; ++q) {
        const bool me = q == qp;
        rank = me ? cnt[q] : rank;
        cnt[q] += me;
        key[q] += me ? ((K)w << kWorkerBits) : (K)0;
      }
      if (mine) worker_of[i] = p + cm * rank;
      my_min = lane_min();
    }
  }
#pragma unroll
  for (int q = 0; q < KMAX; ++q) {
    const int p = lane + 32 * q;
    if (p < m) { counts[p] = cnt[q]; final_load[p] = (long long)(key[q] >> kWorkerBits); }
  }
}

// Phase 2 with a bonus above the total planning load: an item's home key, lowered by the
// bonus, is negative and so below every other key, so every item stays at home. One warp
// walks the stable order 32 items at a time; items with the same home take consecutive
// ranks in that order (match_any), as the one-at-a-time greedy would place them.
__device__ __forceinline__ void greedy_all_home(const Sorted sorted, const int32_t* __restrict__ loads,
                                                const int32_t* __restrict__ home, int bc, int ic, int n, int m,
                                                int cm, int* counts, long long* final_load,
                                                int32_t* __restrict__ worker_of) {
  const int lane = threadIdx.x & 31;
  for (int p = lane; p < m; p += 32) {
    counts[p] = 0;
    final_load[p] = 0;
  }
  __syncwarp();
  for (int base = 0; base < n; base += 32) {
    const int t = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, t < n);
    if (t < n) {
      const int i = sorted[t];
      const int h = home[i];
      const unsigned peers = __match_any_sync(active, h);
      const unsigned below = peers & ((1u << lane) - 1u);
      worker_of[i] = h + cm * (counts[h] + __popc(below));
      atomicAdd(reinterpret_cast<unsigned long long*>(&final_load[h]),
                (unsigned long long)((long long)loads[i] * bc + ic));
      __syncwarp(active);
      if (below == 0) counts[h] += __popc(peers);
    }
    __syncwarp();
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1) lpt_plan_kernel(
    const int32_t* __restrict__ loads, const int32_t* __restrict__ home, int n_max, const int32_t* n_dev, int m,
    int bonus, int bc, int ic, int32_t* __restrict__ worker_of, int32_t* __restrict__ offsets,
    int32_t* __restrict__ worklist, int64_t* __restrict__ worker_loads, int* err) {
  dbsp::ptx::griddep_wait();  // the loads come from the previous grid
  dbsp::ptx::griddep_launch_dependents();
  // the item count: n_max, or the first *n_dev items when the count lives on the device
  const int n = n_dev ? min(n_max, max(0, *n_dev)) : n_max;
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ PlanShared sh;
  __shared__ int counts[DBSP_MAX_WORKERS + 1];
  __shared__ long long final_load[DBSP_MAX_WORKERS];
  __shared__ long long keys[2][DBSP_MAX_WORKERS];
  const int tid = threadIdx.x, lane = tid & 31;

  // ---- phase 0: validate and find the load range
  if (tid == 0) { sh.min_load = INT_MAX; sh.max_load = INT_MIN; sh.bad_home = 0; sh.total_load = 0; }
  __syncthreads();
  int lmin = INT_MAX, lmax = INT_MIN, badh = 0;
  unsigned long long tot = 0;
  const bool vec4 = ((reinterpret_cast<uintptr_t>(loads) | reinterpret_cast<uintptr_t>(home)) & 15u) == 0;
  const int n4 = vec4 ? n / 4 : 0;  // items [0, 4 n4) read as int4
  const bool deep = n >= kDeepItems;
  // a large plan reads its loads (and homes) from DRAM in several rounds of reads in
  // flight: one bulk L2 prefetch of each array first pays the latency once
  if (deep && vec4 && tid == 0) {
    constexpr uint32_t kChunk = 1u << 16;
    const uint32_t bytes = (uint32_t)n4 * 16u;
    for (uint32_t o = 0; o < bytes; o += kChunk) {
      const uint32_t len = min(kChunk, bytes - o);
      dbsp::ptx::bulk_prefetch_l2(reinterpret_cast<const char*>(loads) + o, len);
      if (home) dbsp::ptx::bulk_prefetch_l2(reinterpret_cast<const char*>(home) + o, len);
    }
  }
  auto validate = [&](auto depth) {
    constexpr int kU = decltype(depth)::value;
    for (int base = tid; base < n4; base += kU * kThreads) {
      int4 v[kU], hv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kThreads;
        v[u] = i < n4 ? __ldg(reinterpret_cast<const int4*>(loads) + i) : make_int4(0, 0, 0, 0);
        hv[u] = (home && i < n4) ? __ldg(reinterpret_cast<const int4*>(home) + i) : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (base + u * kThreads < n4) {
          const int w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          const int h4[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            lmin = min(lmin, w4[e]); lmax = max(lmax, w4[e]);
            tot += (unsigned long long)max(w4[e], 0) * (unsigned long long)bc + (unsigned long long)ic;
            badh |= (h4[e] < 0 || h4[e] >= m);
          }
        }
      }
    }
    for (int base = 4 * n4 + tid; base < n; base += kU * kThreads) {
      int v[kU], hv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kThreads;
        v[u] = i < n ? __ldg(loads + i) : 0;
        hv[u] = (home && i < n) ? __ldg(home + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (base + u * kThreads < n) {
          const int w = v[u];
          lmin = min(lmin, w); lmax = max(lmax, w);
          tot += (unsigned long long)max(w, 0) * (unsigned long long)bc + (unsigned long long)ic;
          badh |= (hv[u] < 0 || hv[u] >= m);
        }
      }
    }
  };
  if (deep)
    validate(Depth<8>{});
  else
    validate(Depth<4>{});
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane == 0) atomicAdd(&sh.total_load, tot);  // one atomic per warp
  atomicMin(&sh.min_load, lmin);
  atomicMax(&sh.max_load, lmax);
  if (badh) atomicOr(&sh.bad_home, 1);
  __syncthreads();
  const bool ok_vals = n == 0 || (sh.min_load >= 0 && !sh.bad_home);
  const int max_load = n ? sh.max_load : 0;
  // planning loads load * bc + ic must stay within int
  const bool ok_cost = (long long)max_load * bc + ic < (1LL << 31);
  const bool staged = n <= kStagedMaxItems && max_load <= kStagedMaxLoad;
  const bool counting = max_load <= kMaxLoadCounting;
  if (!ok_vals || !ok_cost || (!counting && n > kMaxItemsCompare)) {
    if (tid == 0) dbsp::report(err, ok_vals ? DBSP_ERR_UNSUPPORTED : DBSP_ERR_INVALID_ARG);
    for (int p = tid; p <= m; p += kThreads) offsets[p] = 0;
    return;
  }
  const int nbins = max_load + 1;
  // worker_of holds worker + cm * (rank within worker) until the CSR scatter: cm = 1024
  // (a shift) whenever ranks stay below 2^21, else m
  const int cm = n < (1 << 21) ? DBSP_MAX_WORKERS : m;

  // ---- phase 1: stable order by (load desc, id asc)
  Sorted sorted{nullptr, worklist};
  const uint16_t* sload = nullptr;  // load of each sorted position (staged, n <= 22528)
  const int* bin_end = nullptr;  // bin_end[b] = one past the last sorted position of bin b
  if (staged) {
    // 8 warps each take a contiguous id segment: per-warp histograms, a scan over
    // (bin, warp), then each warp scatters its segment in id order (stable)
    uint16_t* order = reinterpret_cast<uint16_t*>(dyn);
    // the order takes bytes [0, 2n); the loads of the sorted positions, when n <= 22528,
    // [45056, 45056 + 2n); the bin cursor and the per-warp histograms start at 90112
    int* cursor = reinterpret_cast<int*>(dyn + 2 * kStagedMaxItems);  // [nbins + 1]
    int* whist = cursor + (nbins + 1);                    // [8][nbins]
    const int warp = tid >> 5;
    constexpr int kWarps = kThreads / 32;
    const int seg = (n + kWarps - 1) / kWarps;
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    for (int b = tid; b < kWarps * nbins; b += kThreads) whist[b] = 0;
    __syncthreads();
    // the segment [lo, hi): its 16-byte-aligned middle as int4, the ends item by item
    const int vlo = vec4 ? min(hi, (lo + 3) & ~3) : hi, vhi = vec4 ? max(vlo, hi & ~3) : hi;
    for (int i = lo + lane; i < vlo; i += 32) atomicAdd(&whist[warp * nbins + (max_load - __ldg(loads + i))], 1);
    for (int i = vhi + lane; i < hi; i += 32) atomicAdd(&whist[warp * nbins + (max_load - __ldg(loads + i))], 1);
    auto histogram = [&](auto depth) {
      constexpr int kU = decltype(depth)::value;
      for (int base = vlo / 4 + lane; base < vhi / 4; base += 32 * kU) {
        int4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
          v[u] = base + 32 * u < vhi / 4 ? __ldg(reinterpret_cast<const int4*>(loads) + base + 32 * u)
                                         : make_int4(-1, -1, -1, -1);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (v[u].x >= 0) {
            atomicAdd(&whist[warp * nbins + (max_load - v[u].x)], 1);
            atomicAdd(&whist[warp * nbins + (max_load - v[u].y)], 1);
            atomicAdd(&whist[warp * nbins + (max_load - v[u].z)], 1);
            atomicAdd(&whist[warp * nbins + (max_load - v[u].w)], 1);
          }
        }
      }
    };
    if (deep)
      histogram(Depth<8>{});
    else
      histogram(Depth<4>{});
    __syncthreads();
    for (int b = tid; b <= nbins; b += kThreads) {
      int t = 0;
      if (b < nbins)
        for (int w = 0; w < kWarps; ++w) t += whist[w * nbins + b];
      cursor[b] = t;
    }
    __syncthreads();
    block_exclusive_scan(cursor, nbins + 1, sh.scan);
    for (int b = tid; b < nbins; b += kThreads) {
      int run = cursor[b];
      for (int w = 0; w < kWarps; ++w) { const int t = whist[w * nbins + b]; whist[w * nbins + b] = run; run += t; }
    }
    __syncthreads();
    int* mine = whist + warp * nbins;
    // the loads of each sorted position as well, when they fit beside the order
    uint16_t* sl = n <= kStagedMaxItems / 2 ? reinterpret_cast<uint16_t*>(dyn + kStagedMaxItems) : nullptr;
    // groups of kC chunks of 32 ids; the next group's loads are read while this one is placed
    constexpr int kC = 8;
    auto fetch = [&](int base0, int (&x)[kC]) {
#pragma unroll
      for (int u = 0; u < kC; ++u) {
        const int i = base0 + 32 * u + lane;
        x[u] = i < hi ? __ldg(loads + i) : -1;
      }
    };
    int v[kC];
    fetch(lo, v);
    for (int base0 = lo; base0 < hi; base0 += 32 * kC) {
      int nv[kC];
      fetch(base0 + 32 * kC, nv);
      // a group whose ids all carry one load (a head of equal row loads) fills consecutive
      // positions of its bin at once
      const int v0 = __shfl_sync(0xffffffffu, v[0], 0);  // (id base0 < hi)
      bool one = true;
#pragma unroll
      for (int u = 0; u < kC; ++u) one &= v[u] == v0 || base0 + 32 * u + lane >= hi;
      if (__all_sync(0xffffffffu, one)) {
        const int bin = max_load - v0;
        const int pos0 = mine[bin];
#pragma unroll
        for (int u = 0; u < kC; ++u) {
          const int i = base0 + 32 * u + lane;
          if (i < hi) {
            order[pos0 + 32 * u + lane] = (uint16_t)i;
            if (sl) sl[pos0 + 32 * u + lane] = (uint16_t)v0;
          }
        }
        __syncwarp();
        if (lane == 0) mine[bin] = pos0 + min(32 * kC, hi - base0);
        __syncwarp();
      } else {
#pragma unroll
        for (int u = 0; u < kC; ++u) {
          const int i = base0 + 32 * u + lane;
          const unsigned active = __ballot_sync(0xffffffffu, i < hi);
          if (i < hi) {
            const int bin = max_load - v[u];
            const unsigned peers = __match_any_sync(active, bin);
            const unsigned below = peers & ((1u << lane) - 1);
            const int pos = mine[bin] + __popc(below);
            order[pos] = (uint16_t)i;
            if (sl) sl[pos] = (uint16_t)v[u];
            __syncwarp(active);
            if (below == 0) mine[bin] += __popc(peers);
          }
          __syncwarp();
        }
      }
#pragma unroll
      for (int u = 0; u < kC; ++u) v[u] = nv[u];
    }
    sload = sl;
    sorted = Sorted{order, nullptr};
    bin_end = cursor + 1;
  } else if (counting) {
    int* cursor = reinterpret_cast<int*>(dyn);
    for (int b = tid; b <= nbins; b += kThreads) cursor[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) atomicAdd(&cursor[max_load - loads[i]], 1);
    __syncthreads();
    block_exclusive_scan(cursor, nbins + 1, sh.scan);
    if (tid < 32) {  // stable scatter in id order, 32 ids at a time, into the worklist
      for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const unsigned active = __ballot_sync(0xffffffffu, i < n);
        if (i < n) {
          const int bin = max_load - loads[i];
          const unsigned peers = __match_any_sync(active, bin);
          const unsigned below = peers & ((1u << lane) - 1);
          worklist[cursor[bin] + __popc(below)] = i;
          __syncwarp(active);
          if (below == 0) cursor[bin] += __popc(peers);
        }
        __syncwarp();
      }
    }
    bin_end = cursor;  // after the scatter each cursor is the end of its bin
  } else {
    int* w_s = reinterpret_cast<int*>(dyn);
    for (int i = tid; i < n; i += kThreads) w_s[i] = loads[i];
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const int wi = w_s[i];
      int rank = 0;
      for (int j = 0; j < n; ++j) {
        const int wj = w_s[j];
        rank += (wj > wi) || (wj == wi && j < i);
      }
      worklist[rank] = i;
    }
  }
  __syncthreads();

  // ---- phase 2: the greedy
  const long long wmax = (long long)max_load * bc + ic;  // the largest planning load
  int ring_R = 2;
  while (ring_R < 2 * wmax + 1 && ring_R < (1 << 20)) ring_R <<= 1;
  const int wpb = (m + 31) >> 5;
  const bool ring = staged && ring_R <= kRingMax && (long long)ring_R * wpb <= kRingWords &&
                    (long long)n * wmax < (1LL << 31);
  if (home != nullptr && bonus > 0 && (unsigned long long)bonus > sh.total_load) {
    if (tid < 32) greedy_all_home(sorted, loads, home, bc, ic, n, m, cm, counts, final_load, worker_of);
  } else if (counting && (home == nullptr || bonus == 0) && ring) {
    // without staged loads, the table of runs (non-empty load bins, heaviest first) in the
    // key array, which this path does not use: one warp compacts the bins by ballots
    int* run = sload ? nullptr : reinterpret_cast<int*>(keys[0]);
    if (run && tid < 32) {
      int nr = 0;
      for (int b0 = 0; b0 < nbins; b0 += 32) {
        const int b = b0 + lane;
        const int e = b < nbins ? bin_end[b] : 0;
        const bool used = b < nbins && e > (b == 0 ? 0 : bin_end[b - 1]);
        const unsigned ballot = __ballot_sync(0xffffffffu, used);
        if (used) run[nr + __popc(ballot & ((1u << lane) - 1u))] = (e << kRunLoadBits) | (max_load - b);
        nr += __popc(ballot);
      }
    }
    __syncthreads();
    constexpr int WPT = (KMAX * 32 + kThreads - 1) / kThreads;
    if (!greedy_sorted<WPT>(loads, sorted.smem, sload, bin_end, max_load, run, n, m, cm, bc, ic, ring_R,
                       reinterpret_cast<uint32_t*>(dyn + kRingOff), reinterpret_cast<int*>(dyn + kPreOff),
                       reinterpret_cast<int*>(dyn + kCntOff), reinterpret_cast<int*>(dyn + kLwOff),
                       reinterpret_cast<unsigned long long*>(dyn + kAOff), counts, final_load, worker_of, sh.scan)) {
      if (tid == 0) dbsp::report(err, DBSP_ERR_UNSUPPORTED);
      for (int p = tid; p <= m; p += kThreads) offsets[p] = 0;
      return;
    }
  } else if (counting && (home == nullptr || bonus == 0)) {
    // LPT keeps every worker within max_load of the average, so the final worker load is
    // below total / m + max_load; 32-bit keys (load < 2^21) halve the shared-memory
    // traffic of the batch merges whenever that bound allows
    constexpr int KT = (KMAX * 32 + kThreads - 1) / kThreads;
    const bool key32 = sh.total_load / (unsigned long long)m + (unsigned long long)max_load * bc + ic < (1ull << 20);
    if (key32)
      greedy_batched<KT, uint32_t>(sorted, bin_end, nbins, max_load, n, m, cm, bc, ic,
                                   reinterpret_cast<uint32_t*>(keys[0]), counts, final_load, worker_of, sh.scan);
    else
      greedy_batched<KT, long long>(sorted, bin_end, nbins, max_load, n, m, cm, bc, ic, keys[0], counts, final_load,
                                    worker_of, sh.scan);
  } else if (tid < 32) {
    // a worker takes an item only while its key, lowered by at most the bonus, is the
    // smallest: every load stays below total / m + the largest planning load + bonus
    const bool key32 =
        sh.total_load / (unsigned long long)m + (unsigned long long)max_load * bc + ic + (unsigned)bonus < (1ull << 19);
    if (key32)
      greedy_serial<KMAX, int>(sorted, loads, home, bonus, bc, ic, n, m, cm, counts, final_load, worker_of);
    else
      greedy_serial<KMAX, long long>(sorted, loads, home, bonus, bc, ic, n, m, cm, counts, final_load, worker_of);
  }
  __syncthreads();

  // ---- phase 3: CSR offsets and scatter
  if (tid == 0) counts[m] = 0;
  __syncthreads();
  block_exclusive_scan(counts, m + 1, sh.scan);
  for (int p = tid; p <= m; p += kThreads) offsets[p] = counts[p];
  if (worker_loads)
    for (int p = tid; p < m; p += kThreads) worker_loads[p] = final_load[p];
  const bool wvec = (reinterpret_cast<uintptr_t>(worker_of) & 15u) == 0;
  const int nw4 = wvec ? n / 4 : 0;
  // The worklist is a scatter (item i to offsets[p] + rank). With the greedy done, the
  // dynamic shared memory is free: for large plans that fit, the worklist is assembled
  // there and written out with coalesced stores instead of one scattered global store
  // per item (imbalance workload, 40,960 items: 180 -> 166 us).
  int* ws = n >= 8192 && (size_t)n * sizeof(int) <= kDynBytes ? reinterpret_cast<int*>(dyn) : nullptr;
  int32_t* wdst = ws ? ws : worklist;
  auto scatter = [&](auto depth) {
    constexpr int kU = decltype(depth)::value;
    for (int base = tid; base < nw4; base += kU * kThreads) {
      int4 c4[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        c4[u] = base + u * kThreads < nw4 ? reinterpret_cast<const int4*>(worker_of)[base + u * kThreads]
                                          : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i4 = base + u * kThreads;
        if (i4 < nw4) {
          const int cc[4] = {c4[u].x, c4[u].y, c4[u].z, c4[u].w};
          int pp[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int p = cm == DBSP_MAX_WORKERS ? (cc[e] & (DBSP_MAX_WORKERS - 1)) : cc[e] % m;
            const int rank = cm == DBSP_MAX_WORKERS ? (cc[e] >> 10) : cc[e] / m;
            wdst[counts[p] + rank] = 4 * i4 + e;
            pp[e] = p;
          }
          reinterpret_cast<int4*>(worker_of)[i4] = make_int4(pp[0], pp[1], pp[2], pp[3]);
        }
      }
    }
    for (int base = 4 * nw4 + tid; base < n; base += kU * kThreads) {
      int code[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) code[u] = base + u * kThreads < n ? worker_of[base + u * kThreads] : 0;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kThreads;
        if (i < n) {
          const int p = cm == DBSP_MAX_WORKERS ? (code[u] & (DBSP_MAX_WORKERS - 1)) : code[u] % m;
          const int rank = cm == DBSP_MAX_WORKERS ? (code[u] >> 10) : code[u] / m;
          wdst[counts[p] + rank] = i;
          worker_of[i] = p;
        }
      }
    }
  };
  if (deep)
    scatter(Depth<8>{});
  else
    scatter(Depth<4>{});
  if (ws) {
    __syncthreads();
    const bool lvec = (reinterpret_cast<uintptr_t>(worklist) & 15u) == 0;
    const int nl4 = lvec ? n / 4 : 0;
    for (int q = tid; q < nl4; q += kThreads) reinterpret_cast<int4*>(worklist)[q] = reinterpret_cast<const int4*>(ws)[q];
    for (int q = 4 * nl4 + tid; q < n; q += kThreads) worklist[q] = ws[q];
  }
}

template <int KMAX>
int launch(const int32_t* loads, const int32_t* home, int n, const int32_t* n_dev, int m, int bonus, int bc, int ic,
           int32_t* worker_of, int32_t* offsets, int32_t* worklist, int64_t* worker_loads, int* err,
           cudaStream_t s) {
  auto kernel = lpt_plan_kernel<KMAX>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynBytes);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(lpt_plan)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kDynBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {dbsp::overlap_previous_grid()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, loads, home, n, n_dev, m, bonus, bc, ic, worker_of, offsets, worklist,
                         worker_loads, err);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch lpt_plan");
  return DBSP_OK;
}

}  // namespace

namespace {

int plan_lpt(const int32_t* loads, const int32_t* home, int n_items, const int32_t* n_dev, int n_workers,
             int32_t stay_bonus, int32_t block_cost, int32_t item_cost, int32_t* worker_of, int32_t* worker_offsets,
             int32_t* worklist, int64_t* worker_loads, void* stream) {
  if (n_items < 0 || n_workers < 1 || n_workers > DBSP_MAX_WORKERS || stay_bonus < 0)
    return DBSP_ERR_INVALID_ARG;
  if (block_cost < 1 || block_cost > 65535 || item_cost < 0 || item_cost > (1 << 24)) return DBSP_ERR_INVALID_ARG;
  if ((long long)n_items * n_workers >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (!worker_offsets) return DBSP_ERR_INVALID_ARG;
  if (n_items > 0 && (!loads || !worker_of || !worklist)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  int* err = dbsp::error_word(dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int m = n_workers;
#define DBSP_PLAN_CASE(K)                                                                                        \
  return launch<K>(loads, home, n_items, n_dev, m, stay_bonus, block_cost, item_cost, worker_of, worker_offsets, \
                   worklist, worker_loads, err, s)
  if (m <= 32) DBSP_PLAN_CASE(1);
  if (m <= 64) DBSP_PLAN_CASE(2);
  if (m <= 128) DBSP_PLAN_CASE(4);
  if (m <= 256) DBSP_PLAN_CASE(8);
  if (m <= 512) DBSP_PLAN_CASE(16);
  DBSP_PLAN_CASE(32);
#undef DBSP_PLAN_CASE
}

}  // namespace

extern "C" int dbsp_plan_lpt_cost(const int32_t* loads, const int32_t* home, int n_items, int n_workers,
                                  int32_t stay_bonus, int32_t block_cost, int32_t item_cost, int32_t* worker_of,
                                  int32_t* worker_offsets, int32_t* worklist, int64_t* worker_loads,
                                  void* stream) {
  return plan_lpt(loads, home, n_items, nullptr, n_workers, stay_bonus, block_cost, item_cost, worker_of,
                  worker_offsets, worklist, worker_loads, stream);
}

extern "C" int dbsp_plan_lpt_cost_n(const int32_t* loads, const int32_t* n_items_dev, int n_items_max,
                                    int n_workers, int32_t block_cost, int32_t item_cost, int32_t* worker_of,
                                    int32_t* worker_offsets, int32_t* worklist, int64_t* worker_loads,
                                    void* stream) {
  if (!n_items_dev) return DBSP_ERR_INVALID_ARG;
  return plan_lpt(loads, nullptr, n_items_max, n_items_dev, n_workers, 0, block_cost, item_cost, worker_of,
                  worker_offsets, worklist, worker_loads, stream);
}

extern "C" int dbsp_plan_lpt(const int32_t* loads, const int32_t* home, int n_items, int n_workers,
                             int32_t stay_bonus, int32_t* worker_of, int32_t* worker_offsets,
                             int32_t* worklist, int64_t* worker_loads, void* stream) {
  return plan_lpt(loads, home, n_items, nullptr, n_workers, stay_bonus, 1, 0, worker_of, worker_offsets,
                  worklist, worker_loads, stream);
}
