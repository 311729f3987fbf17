// Splitting heavy items into pieces along their KV blocks: the unit table.
//
// db-SP blog, scenario 1: the greedy cannot balance perfectly, partly because an
// item's load cannot be divided; the page's closing remark points at splitting the
// load further. An item whose load L exceeds T becomes k = min(ceil(L / T), P) pieces;
// piece j takes the row's dense blocks of rank [floor(j L / k), floor((j + 1) L / k))
// (the attention producer finds them while it scans the row), and is attended as a
// partial (O, m, l) written to its own slot; dbsp_merge_pieces combines the pieces.
//
// Unit table: first the whole items in item order, then the pieces of the split items
// in (item, j) order at unit n_whole + slot; unit_pk packs j | k << 16. One CTA:
//   pass 0  check the loads, their total (T <= 0 selects T = ceil(ceil(total / m) / 2));
//   pass 1  per thread, over a contiguous range of items: whole items, split items and
//           pieces; block scans of the three counts;
//   pass 2  every item writes its units at the scanned positions.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

struct SplitShared {
  unsigned long long total;
  int bad;
};

__device__ __forceinline__ int pieces_of(int load, int t, int p) {
  return load <= t ? 1 : min((int)(((long long)load + t - 1) / t), p);
}

// Exclusive scan of one int per thread across the CTA; returns this thread's base and
// sets *total. `ws` holds one int per warp.
__device__ int cta_exclusive_scan(int x, int* ws, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < kWarps ? ws[lane] : 0;
    int wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) ws[lane] = wi - v;
    if (lane == kWarps - 1) ws[kWarps] = wi;
  }
  __syncthreads();
  const int base = ws[warp] + incl - x;
  *total = ws[kWarps];
  __syncthreads();
  return base;
}

__global__ void __launch_bounds__(kThreads, 1) split_plan_kernel(
    const int32_t* __restrict__ loads, int n, int t_in, int p_max, int m, int max_slots,
    int32_t* __restrict__ unit_item, int32_t* __restrict__ unit_pk, int32_t* __restrict__ unit_slot,
    int32_t* __restrict__ unit_load, int32_t* __restrict__ split_item, int32_t* __restrict__ split_off,
    int32_t* __restrict__ counts, int* err) {
  __shared__ SplitShared sh;
  __shared__ int ws[kWarps + 1];
  const int tid = threadIdx.x;
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  if (tid == 0) {
    sh.total = 0;
    sh.bad = 0;
  }
  __syncthreads();
  // pass 0: validity and total load
  unsigned long long tot = 0;
  int bad = 0;
  for (int i = lo; i < hi; ++i) {
    const int w = loads[i];
    bad |= w < 0;
    tot += (unsigned long long)max(w, 0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if ((tid & 31) == 0) atomicAdd(&sh.total, tot);
  if (bad) atomicOr(&sh.bad, 1);
  __syncthreads();
  if (sh.bad) {
    if (tid == 0) {
      dbsp::report(err, DBSP_ERR_INVALID_ARG);
      counts[0] = counts[1] = counts[2] = counts[3] = 0;
      counts[4] = 0;
      split_off[0] = 0;
    }
    return;
  }
  long long t = t_in;
  if (t <= 0) {  // half the mean load per worker, rounded up, at least 1
    const long long mean = (long long)((sh.total + (unsigned long long)m - 1) / (unsigned long long)m);
    t = max(1LL, (mean + 1) / 2);
  }
  const int T = (int)min(t, (long long)INT_MAX);
  // pass 1: counts per thread, then the scans
  int cw = 0, cs = 0, cl = 0;
  for (int i = lo; i < hi; ++i) {
    const int k = pieces_of(loads[i], T, p_max);
    if (k == 1) ++cw;
    else { ++cs; cl += k; }
  }
  int n_whole, n_split, n_slots;
  int bw = cta_exclusive_scan(cw, ws, &n_whole);
  int bs = cta_exclusive_scan(cs, ws, &n_split);
  int bl = cta_exclusive_scan(cl, ws, &n_slots);
  if (n_slots > max_slots) {
    if (tid == 0) {
      dbsp::report(err, DBSP_ERR_UNSUPPORTED);
      counts[0] = counts[1] = counts[2] = counts[3] = 0;
      counts[4] = T;
      split_off[0] = 0;
    }
    return;
  }
  // pass 2: the units
  for (int i = lo; i < hi; ++i) {
    const int L = loads[i];
    const int k = pieces_of(L, T, p_max);
    if (k == 1) {
      const int u = bw++;
      unit_item[u] = i;
      unit_pk[u] = 1 << 16;
      unit_slot[u] = -1;
      unit_load[u] = L;
    } else {
      const int si = bs++, slot0 = bl;
      bl += k;
      split_item[si] = i;
      split_off[si] = slot0;
      for (int j = 0; j < k; ++j) {
        const int u = n_whole + slot0 + j;
        unit_item[u] = i;
        unit_pk[u] = j | (k << 16);
        unit_slot[u] = slot0 + j;
        unit_load[u] = (int)(((long long)(j + 1) * L) / k - ((long long)j * L) / k);
      }
    }
  }
  if (tid == 0) {
    split_off[n_split] = n_slots;
    counts[0] = n_whole + n_slots;
    counts[1] = n_whole;
    counts[2] = n_split;
    counts[3] = n_slots;
    counts[4] = T;
  }
}

}  // namespace

extern "C" int dbsp_split_plan(const int32_t* loads, int n_items, int n_workers, int32_t max_piece_load,
                               int32_t max_pieces, int32_t max_slots, int32_t* unit_item, int32_t* unit_pk,
                               int32_t* unit_slot, int32_t* unit_load, int32_t* split_item,
                               int32_t* split_off, int32_t* counts, void* stream) {
  if (n_items < 0 || n_workers < 1 || max_pieces < 1 || max_pieces > 1024 || max_slots < 0)
    return DBSP_ERR_INVALID_ARG;
  if ((long long)n_items * max_pieces >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (!counts || !split_off) return DBSP_ERR_INVALID_ARG;
  if (n_items > 0 && (!loads || !unit_item || !unit_pk || !unit_slot || !unit_load || !split_item))
    return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  split_plan_kernel<<<1, kThreads, 0, s>>>(loads, n_items, max_piece_load, max_pieces, n_workers, max_slots,
                                           unit_item, unit_pk, unit_slot, unit_load, split_item, split_off,
                                           counts, dbsp::error_word(dev));
  DBSP_LAUNCH_CHECK("launch split_plan");
  return DBSP_OK;
}
