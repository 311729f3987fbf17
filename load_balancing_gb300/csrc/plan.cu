// LPT planning with a stay-in-place bonus, on the device, bit-exact.
//
// db-SP blog, scenario 1: the longest remaining item goes to the least-loaded
// worker (LPT, the greedy for identical-machines scheduling). db-SP blog,
// scenario 2, third bullet: an item placed on its original worker counts as
// lighter when the worker is chosen. Readings: equal loads are taken by ascending
// id, ties between workers go to the lowest index, the bonus enters only the
// choice and the worker accrues the item's true load.
//
// One CTA of 256 threads:
//   phase 0  check loads/home, find the load range;
//   phase 1  stable order by (load desc, id asc): a counting sort through a
//            shared-memory histogram (loads <= 32767), else rank-by-comparison
//            (n <= 16384). The order is written into `worklist`;
//   phase 2  the greedy, one warp: every lane keeps the loads of workers
//            lane, lane+32, ... in registers as packed keys (load << 11 | worker),
//            so (load, worker) order is plain int64 order; the warp minimum is two
//            redux.sync reductions (high word, then low word among the tied);
//            `worker_of[i]` temporarily holds worker + m * (rank within worker);
//   phase 3  CSR offsets by a block scan of the per-worker counts, then the
//            scatter of every item to offsets[worker] + rank.
// The output arrays are the only global working storage.
#include <algorithm>
#include <climits>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxLoadCounting = 32767;
constexpr int kMaxItemsCompare = 16384;
constexpr int kWorkerBits = 11;  // worker index < 2048 in the packed key
constexpr long long kKeyNone = LLONG_MAX;

struct PlanShared {
  int min_load, max_load, bad_home;
  int scan[kThreads / 32 + 1];
};

// Exclusive scan over `n` ints in shared memory `a` (in place). Returns the total.
__device__ int block_exclusive_scan(int* a, int n, int* warp_sums) {
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
    warp_sums[kThreads / 32] = run;
  }
  __syncthreads();
  int run = warp_sums[warp] + x - s;
  for (int j = lo; j < hi; ++j) { const int t = a[j]; a[j] = run; run += t; }
  const int total = warp_sums[kThreads / 32];
  __syncthreads();
  return total;
}

template <int KMAX>
__device__ __forceinline__ long long lane_minimum(const long long (&key)[KMAX]) {
  long long m = key[0];
#pragma unroll
  for (int q = 1; q < KMAX; ++q) m = key[q] < m ? key[q] : m;
  return m;
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1) lpt_plan_kernel(
    const int32_t* __restrict__ loads, const int32_t* __restrict__ home, int n, int m,
    int bonus, int32_t* __restrict__ worker_of, int32_t* __restrict__ offsets,
    int32_t* __restrict__ worklist, int64_t* __restrict__ worker_loads, int* err) {
  extern __shared__ int dyn[];  // histogram / cursor, or a copy of the loads
  __shared__ PlanShared sh;
  __shared__ int counts[DBSP_MAX_WORKERS + 1];
  __shared__ long long final_load[DBSP_MAX_WORKERS];
  const int tid = threadIdx.x, lane = tid & 31;

  // ---- phase 0: validate and find the load range
  if (tid == 0) { sh.min_load = INT_MAX; sh.max_load = INT_MIN; sh.bad_home = 0; }
  __syncthreads();
  int lmin = INT_MAX, lmax = INT_MIN, badh = 0;
  for (int i = tid; i < n; i += kThreads) {
    const int w = loads[i];
    lmin = min(lmin, w); lmax = max(lmax, w);
    if (home) { const int h = home[i]; badh |= (h < 0 || h >= m); }
  }
  atomicMin(&sh.min_load, lmin);
  atomicMax(&sh.max_load, lmax);
  if (badh) atomicOr(&sh.bad_home, 1);
  __syncthreads();
  const bool ok_vals = n == 0 || (sh.min_load >= 0 && !sh.bad_home);
  const bool counting = n == 0 || sh.max_load <= kMaxLoadCounting;
  if (!ok_vals || (!counting && n > kMaxItemsCompare)) {
    if (tid == 0) dbsp::report(err, ok_vals ? DBSP_ERR_UNSUPPORTED : DBSP_ERR_INVALID_ARG);
    for (int p = tid; p <= m; p += kThreads) offsets[p] = 0;
    return;
  }
  const int max_load = n ? sh.max_load : 0;

  // ---- phase 1: stable order by (load desc, id asc) into worklist
  if (counting) {
    int* cursor = dyn;  // bins are indexed by (max_load - load): descending loads first
    const int nbins = max_load + 1;
    for (int b = tid; b < nbins; b += kThreads) cursor[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) atomicAdd(&cursor[max_load - loads[i]], 1);
    __syncthreads();
    block_exclusive_scan(cursor, nbins, sh.scan);
    if (tid < 32) {  // stable scatter in id order, 32 ids at a time
      for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const unsigned active = __ballot_sync(0xffffffffu, i < n);
        if (i < n) {
          const int bin = max_load - loads[i];
          const unsigned peers = __match_any_sync(active, bin);
          const int pos = cursor[bin] + __popc(peers & ((1u << lane) - 1));
          worklist[pos] = i;
          __syncwarp(active);
          if ((peers & ((1u << lane) - 1)) == 0) cursor[bin] += __popc(peers);
        }
        __syncwarp();
      }
    }
  } else {
    int* w_s = dyn;
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

  // ---- phase 2: the greedy (warp 0)
  if (tid < 32) {
    long long key[KMAX];
    int cnt[KMAX];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
      const int p = lane + 32 * q;
      key[q] = p < m ? (long long)p : kKeyNone;  // load 0, worker p
      cnt[q] = 0;
    }
    long long my_min = lane_minimum(key);
    const long long bonus_key = (long long)bonus << kWorkerBits;
    for (int base = 0; base < n; base += 32) {
      const int t = base + lane;
      int my_i = 0, my_w = 0, my_h = -1;
      if (t < n) {
        my_i = worklist[t];
        my_w = loads[my_i];
        if (home) my_h = home[my_i];
      }
      const int chunk = min(32, n - base);
      for (int s = 0; s < chunk; ++s) {
        const int i = __shfl_sync(0xffffffffu, my_i, s);
        const int w = __shfl_sync(0xffffffffu, my_w, s);
        const int h = __shfl_sync(0xffffffffu, my_h, s);
        long long cand = my_min;
        if (h >= 0 && (h & 31) == lane) {
          long long kh = kKeyNone;
#pragma unroll
          for (int q = 0; q < KMAX; ++q) if (q == (h >> 5)) kh = key[q];
          kh -= bonus_key;
          cand = kh < cand ? kh : cand;
        }
        const int hi = (int)(cand >> 32);
        const int min_hi = __reduce_min_sync(0xffffffffu, hi);
        const unsigned lo = hi == min_hi ? (unsigned)(cand & 0xffffffffu) : 0xffffffffu;
        const unsigned min_lo = __reduce_min_sync(0xffffffffu, lo);
        const int p = (int)(min_lo & ((1u << kWorkerBits) - 1));
        if ((p & 31) == lane) {
          const int qp = p >> 5;
          int rank = 0;
#pragma unroll
          for (int q = 0; q < KMAX; ++q) {
            if (q == qp) { key[q] += (long long)w << kWorkerBits; rank = cnt[q]; cnt[q] += 1; }
          }
          worker_of[i] = p + m * rank;
          my_min = lane_minimum(key);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
      const int p = lane + 32 * q;
      if (p < m) { counts[p] = cnt[q]; final_load[p] = key[q] >> kWorkerBits; }
    }
  }
  __syncthreads();

  // ---- phase 3: CSR offsets and scatter
  if (tid == 0) counts[m] = 0;
  __syncthreads();
  block_exclusive_scan(counts, m + 1, sh.scan);
  for (int p = tid; p <= m; p += kThreads) offsets[p] = counts[p];
  if (worker_loads)
    for (int p = tid; p < m; p += kThreads) worker_loads[p] = final_load[p];
  for (int i = tid; i < n; i += kThreads) {
    const int code = worker_of[i];
    const int p = code % m, rank = code / m;
    worklist[counts[p] + rank] = i;
    worker_of[i] = p;
  }
}

template <int KMAX>
int launch(const int32_t* loads, const int32_t* home, int n, int m, int bonus, int32_t* worker_of,
           int32_t* offsets, int32_t* worklist, int64_t* worker_loads, int* err, cudaStream_t s) {
  const size_t smem = sizeof(int) * (size_t)std::max(kMaxLoadCounting + 1, kMaxItemsCompare);
  auto kernel = lpt_plan_kernel<KMAX>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(lpt_plan)");
  kernel<<<1, kThreads, smem, s>>>(loads, home, n, m, bonus, worker_of, offsets, worklist,
                                   worker_loads, err);
  DBSP_LAUNCH_CHECK("launch lpt_plan");
  return DBSP_OK;
}

}  // namespace

extern "C" int dbsp_plan_lpt(const int32_t* loads, const int32_t* home, int n_items, int n_workers,
                             int32_t stay_bonus, int32_t* worker_of, int32_t* worker_offsets,
                             int32_t* worklist, int64_t* worker_loads, void* stream) {
  if (n_items < 0 || n_workers < 1 || n_workers > DBSP_MAX_WORKERS || stay_bonus < 0)
    return DBSP_ERR_INVALID_ARG;
  if ((long long)n_items * n_workers >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (!worker_offsets) return DBSP_ERR_INVALID_ARG;
  if (n_items > 0 && (!loads || !worker_of || !worklist)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  int* err = dbsp::error_word(dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int m = n_workers;
#define DBSP_PLAN_CASE(K) \
  return launch<K>(loads, home, n_items, m, stay_bonus, worker_of, worker_offsets, worklist, worker_loads, err, s)
  if (m <= 32) DBSP_PLAN_CASE(1);
  if (m <= 64) DBSP_PLAN_CASE(2);
  if (m <= 128) DBSP_PLAN_CASE(4);
  if (m <= 256) DBSP_PLAN_CASE(8);
  if (m <= 512) DBSP_PLAN_CASE(16);
  DBSP_PLAN_CASE(32);
#undef DBSP_PLAN_CASE
}
