// Mask loads: dense-block counts per Q-block row, per KV-block column and per head.
//
// db-SP blog, scenario 2, first bullet: a Q-block's load is the number of dense
// blocks in its mask row, a KV-block's load the number in its column; scenario 1
// balances whole heads, whose load is the head's total.
//
// Design: a thread-block cluster of up to 8 CTAs per (b, h) head; each CTA counts a
// band of rows. Row loads are exact per CTA and written directly; column partials are
// combined through distributed shared memory (the streaming kernel pushes each rank's
// sums into the rank that owns those columns; the others let rank 0 read every rank's
// partials), so no global scratch or atomics on the outputs are needed and the outputs
// need no prior zeroing. HBM-bound: every mask byte is read once. A causal
// instantiation counts only the blocks on or below the diagonal.
//
// Rows of at most 4096 bytes on a 16-byte aligned mask (every block mask up to 4096
// KV blocks) take the streaming kernel: one thread moves the band through a ring of
// four 16 KB shared-memory stages with bulk asynchronous copies, so 64 KB per CTA is
// in flight without holding it in registers, and all 256 threads count from shared
// memory. Longer rows use 16-byte register loads, and rows whose length or pointer
// does not allow 16-byte access are read byte by byte.
//
// Also here: the KV-block loads summed over heads, and the block mask of each KV shard
// (db-SP blog, scenario 2).
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;
using namespace dbsp::ptx;

namespace {

#ifndef DBSP_LOADS_MAX_CLUSTER
#define DBSP_LOADS_MAX_CLUSTER 8
#endif
constexpr int kThreads = 256;
constexpr int kMaxCluster = DBSP_LOADS_MAX_CLUSTER;  // CTAs per head (above 8: non-portable clusters)
constexpr int kMaxCols = 16384;  // column partials in shared memory: 64 KB
constexpr int kMaxRows = 131072; // row partials of one CTA (1/8 of a head) in shared memory: 64 KB
#ifndef DBSP_LOADS_STAGE_BYTES
#define DBSP_LOADS_STAGE_BYTES 16384
#endif
#ifndef DBSP_LOADS_STAGES
#define DBSP_LOADS_STAGES 4
#endif
constexpr int kStageBytes = DBSP_LOADS_STAGE_BYTES;  // streaming kernel: one ring stage
constexpr int kStages = DBSP_LOADS_STAGES;           // streaming kernel: ring depth
constexpr int kStreamMaxCols = 4096;                 // rows of <= 4096 B: <= 256 units per row
static_assert(kStageBytes >= kStreamMaxCols, "a stage holds at least one row");
static_assert(kStages * kStageBytes >= 16384, "the ring holds the column slots (256 units x 16 ints)");
constexpr int kStageUnits = kStageBytes / (16 * kThreads);  // 16-byte units per thread in a full stage
static_assert(kStageUnits >= 1 && kStageUnits < 128, "stage size");
constexpr size_t kStreamMaxSmem = 200 * 1024;       // streaming kernel: dynamic shared memory cap
#ifdef DBSP_WAIT_TEST
// Test build only (never the product library): stage waits give up after 20 ms, and
// CTA (0, 0) of the streaming kernel leaves out its first stage (neither the arrival nor
// the copy is issued), so that its wait runs out and the drain and cluster teardown run.
constexpr uint64_t kWaitLimitNs = 20000000ull;       // 20 ms per stage wait
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s per stage wait
#endif
constexpr uint64_t kDrainLimitNs = 100000000ull;     // 100 ms per teardown wait

// Number of non-zero bytes in a 32-bit word, as 0x01 flags per byte.
__device__ __forceinline__ uint32_t nonzero_byte_flags(uint32_t x) {
  return ((((x & 0x7f7f7f7fu) + 0x7f7f7f7fu) | x) >> 7) & 0x01010101u;
}

// Causal variant: only the blocks on or below the diagonal (column <= row) count. Keeps
// the bytes of the 16 columns [col0, col0 + 16) of row `row` that satisfy it.
__device__ __forceinline__ uint4 keep_causal(uint4 x, int col0, int row) {
  const int keep = row - col0 + 1;  // columns of the unit at or before the diagonal
  if (keep >= 16) return x;
  if (keep <= 0) return make_uint4(0u, 0u, 0u, 0u);
  auto word_mask = [&](int k) -> uint32_t {
    const int nb = keep - 4 * k;  // bytes kept of word k
    return nb >= 4 ? 0xffffffffu : (nb <= 0 ? 0u : (1u << (8 * nb)) - 1u);
  };
  x.x &= word_mask(0);
  x.y &= word_mask(1);
  x.z &= word_mask(2);
  x.w &= word_mask(3);
  return x;
}

// VEC = 16: each work unit is 16 consecutive mask bytes of one row (uint4 loads);
// VEC = 1: one byte. CAUSAL: count only the blocks on or below the diagonal.
template <int VEC, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) mask_loads_kernel(
    const uint8_t* __restrict__ mask, int nQ, int nK, int rows_per_cta,
    int32_t* __restrict__ row_loads, int32_t* __restrict__ col_loads,
    int32_t* __restrict__ head_loads) {
  extern __shared__ int smem[];
  int* col_part = smem;               // [nK]
  int* row_acc = smem + nK;           // [rows_per_cta]
  __shared__ int cta_total;
  griddep_wait();  // the mask may come from the previous grid
  griddep_launch_dependents();

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int n_ranks = static_cast<int>(cluster.num_blocks());
  const long long head = blockIdx.y;
  const int row0 = rank * rows_per_cta;
  const int row1 = min(nQ, row0 + rows_per_cta);
  const int tid = threadIdx.x;

  for (int j = tid; j < nK; j += kThreads) col_part[j] = 0;
  for (int r = tid; r < rows_per_cta; r += kThreads) row_acc[r] = 0;
  if (tid == 0) cta_total = 0;
  __syncthreads();

  const uint8_t* head_mask = mask + head * nQ * (long long)nK;
  const int cpr = nK / VEC;  // work units per row
  int c0, c_step, r_off, r_step;
  if (cpr <= kThreads) {
    c0 = tid % cpr; c_step = cpr; r_off = tid / cpr; r_step = kThreads / cpr;
  } else {
    c0 = tid; c_step = kThreads; r_off = 0; r_step = 1;
  }
  if (r_off < r_step) {
    for (int c = c0; c < cpr; c += c_step) {
      if (VEC == 16) {
        // per-byte column counters: 4 words of byte-wide counters, flushed before they can pass 255;
        // kUnroll rows are loaded before any is counted, so that many loads are in flight
#ifndef DBSP_LOADS_UNROLL
#define DBSP_LOADS_UNROLL 8
#endif
        constexpr int kUnroll = DBSP_LOADS_UNROLL;
        int cols[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) cols[b] = 0;
        uint32_t acc[4] = {0, 0, 0, 0};
        int pending = 0;
        // a warp that covers 32 units of one row adds its row count once
        const bool warp_row = cpr >= 32 && (cpr % 32) == 0;
        for (int r = row0 + r_off; r < row1; r += kUnroll * r_step) {
          uint4 x[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int ru = r + u * r_step;
            x[u] = ru < row1 ? __ldg(reinterpret_cast<const uint4*>(head_mask + (long long)ru * nK) + c)
                             : make_uint4(0u, 0u, 0u, 0u);
            if (CAUSAL) x[u] = keep_causal(x[u], c * 16, ru);
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int ru = r + u * r_step;
            const uint32_t f0 = nonzero_byte_flags(x[u].x), f1 = nonzero_byte_flags(x[u].y);
            const uint32_t f2 = nonzero_byte_flags(x[u].z), f3 = nonzero_byte_flags(x[u].w);
            acc[0] += f0; acc[1] += f1; acc[2] += f2; acc[3] += f3;
            int cnt = __popc(f0) + __popc(f1) + __popc(f2) + __popc(f3);
            if (warp_row) {
              cnt = __reduce_add_sync(__activemask(), cnt);
              if ((tid & 31) == 0 && cnt && ru < row1) atomicAdd(&row_acc[ru - row0], cnt);
            } else if (cnt) {
              atomicAdd(&row_acc[ru - row0], cnt);
            }
          }
          pending += kUnroll;
          if (pending + kUnroll > 255) {  // the next kUnroll rows could carry a byte counter past 255
#pragma unroll
            for (int b = 0; b < 16; ++b) cols[b] += (acc[b >> 2] >> (8 * (b & 3))) & 0xff;
            acc[0] = acc[1] = acc[2] = acc[3] = 0;
            pending = 0;
          }
        }
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          const int v = cols[b] + ((acc[b >> 2] >> (8 * (b & 3))) & 0xff);
          if (v) atomicAdd(&col_part[c * 16 + b], v);
        }
      } else {
        int col = 0;
        for (int r = row0 + r_off; r < row1; r += r_step) {
          const int nz = (!CAUSAL || c <= r) && __ldg(head_mask + (long long)r * nK + c) != 0;
          col += nz;
          if (nz) atomicAdd(&row_acc[r - row0], 1);
        }
        if (col) atomicAdd(&col_part[c], col);
      }
    }
  }
  __syncthreads();

  int local = 0;
  for (int r = row0 + tid; r < row1; r += kThreads) {
    const int v = row_acc[r - row0];
    row_loads[head * nQ + r] = v;
    local += v;
  }
  local = __reduce_add_sync(0xffffffffu, local);
  if ((tid & 31) == 0 && local) atomicAdd(&cta_total, local);

  cluster.sync();  // every CTA's column partials and total are final
  if (rank == 0) {
    for (int j = tid; j < nK; j += kThreads) {
      int s = 0;
      for (int q = 0; q < n_ranks; ++q) s += cluster.map_shared_rank(col_part, q)[j];
      col_loads[head * nK + j] = s;
    }
    if (tid == 0 && head_loads) {
      int s = 0;
      for (int q = 0; q < n_ranks; ++q) s += *cluster.map_shared_rank(&cta_total, q);
      head_loads[head] = s;
    }
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// Bounded wait on a stage's phase. Returns false on timeout (reported as
// DBSP_ERR_TIMEOUT) or when another thread of the CTA has already given up.
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        dbsp::report(err, DBSP_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Streaming variant for nK % 16 == 0, nK <= kStreamMaxCols and a 16-byte aligned mask.
// Stage i % kStages holds rows [i * chunk_rows, (i + 1) * chunk_rows) of the CTA's band
// (chunk_rows * nK <= kStageBytes). Thread t owns the 16-byte column unit t % (nK / 16)
// and, within a stage, every (256 / (nK / 16))-th row from t / (nK / 16); its per-byte
// column counters therefore stay in registers across the whole band.
template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads) mask_loads_stream_kernel(
    const uint8_t* __restrict__ mask, int nQ, int nK, int rows_per_cta, int chunk_rows,
    int32_t* __restrict__ row_loads, int32_t* __restrict__ col_loads, int32_t* __restrict__ head_loads,
    int* err) {
  extern __shared__ __align__(128) unsigned char dsm[];
  unsigned char* stage = dsm;                                               // [kStages][kStageBytes]
  int* recv = reinterpret_cast<int*>(dsm + kStages * kStageBytes);          // [n_ranks][slice]
  int* row_acc = recv + nK + 4 * kMaxCluster;                               // [rows_per_cta]
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ int cta_total;
  __shared__ int head_part[kMaxCluster];  // rank 0: every rank's total
  __shared__ volatile int abort_flag;
  griddep_wait();  // the mask may come from the previous grid
  griddep_launch_dependents();

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int n_ranks = static_cast<int>(cluster.num_blocks());
  const long long head = blockIdx.y;
  const int row0 = rank * rows_per_cta;
  const int rows = max(0, min(nQ, row0 + rows_per_cta) - row0);
  const int n_chunks = (rows + chunk_rows - 1) / chunk_rows;
  const uint8_t* band = mask + (head * nQ + row0) * (long long)nK;
  const int tid = threadIdx.x;

  auto issue = [&](int i) {  // chunk i into stage i % kStages (thread 0 only)
#ifdef DBSP_WAIT_TEST
    if (i == 0 && blockIdx.x == 0 && blockIdx.y == 0) return;  // the left-out stage
#endif
    const int r = i * chunk_rows;
    const uint32_t bytes = static_cast<uint32_t>(min(chunk_rows, rows - r) * nK);
    const uint32_t bar = smem_u32(&full[i % kStages]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load_g2s(smem_u32(stage + (i % kStages) * kStageBytes), band + (long long)r * nK, bytes, bar);
  };
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbarrier_init();
    for (int i = 0; i < min(kStages, n_chunks); ++i) issue(i);  // the first copies start at once
    cta_total = 0;
    abort_flag = 0;
  }
  for (int r = tid; r < rows_per_cta; r += kThreads) row_acc[r] = 0;
  __syncthreads();
  // first cluster barrier phase: arrive now, wait before the first access to another
  // rank's shared memory (by then every CTA of the cluster has started)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  const int cpr = nK / 16;
  const int c = tid % cpr, r_off = tid / cpr, r_step = kThreads / cpr;
  const bool active = r_off < r_step;
  const bool warp_row = (cpr % 32) == 0;  // a warp's 32 units lie in one row
  // nK a power of two: every thread is active and a full stage gives each exactly
  // kStageUnits units (rows r_off + k * r_step); a row's cpr units are one lane group
  // (cpr < 32) or whole warps (cpr >= 32)
  const bool pow2 = (kThreads % cpr) == 0;
  int cols[16];
#pragma unroll
  for (int b = 0; b < 16; ++b) cols[b] = 0;
  uint32_t acc[4] = {0, 0, 0, 0};  // byte-wide column counters, flushed before they can pass 255
  int pending = 0;
  auto flush_cols = [&]() {
#pragma unroll
    for (int b = 0; b < 16; ++b) cols[b] += (acc[b >> 2] >> (8 * (b & 3))) & 0xff;
    acc[0] = acc[1] = acc[2] = acc[3] = 0;
    pending = 0;
  };
  int failed = -1;  // first chunk whose wait gave up
  for (int i = 0; i < n_chunks; ++i) {
    const bool ok = __all_sync(0xffffffffu, wait_stage(smem_u32(&full[i % kStages]), (i / kStages) & 1,
                                                       &abort_flag, err));
    const unsigned char* src = stage + (i % kStages) * kStageBytes + c * 16;
    const int base = i * chunk_rows;
    const int nr = min(chunk_rows, rows - base);
    if (ok && pow2 && nr == chunk_rows) {
      uint4 x[kStageUnits];
      uint32_t any = 0;
#pragma unroll
      for (int k = 0; k < kStageUnits; ++k) {
        x[k] = *reinterpret_cast<const uint4*>(src + (r_off + k * r_step) * nK);
        if (CAUSAL) x[k] = keep_causal(x[k], c * 16, row0 + base + r_off + k * r_step);
        any |= x[k].x | x[k].y | x[k].z | x[k].w;
      }
      if (!__all_sync(0xffffffffu, (any & 0xfefefefeu) == 0)) {
        // some byte of the warp's units is neither 0 nor 1: reduce every byte to a 0/1 flag
#pragma unroll
        for (int k = 0; k < kStageUnits; ++k) {
          x[k].x = nonzero_byte_flags(x[k].x); x[k].y = nonzero_byte_flags(x[k].y);
          x[k].z = nonzero_byte_flags(x[k].z); x[k].w = nonzero_byte_flags(x[k].w);
        }
      }
#pragma unroll
      for (int k = 0; k < kStageUnits; ++k) {
        acc[0] += x[k].x; acc[1] += x[k].y; acc[2] += x[k].z; acc[3] += x[k].w;
        // byte-wise sum of the four flag words (each byte <= 4), then the sum of its bytes
        int cnt = __dp4a(x[k].x + x[k].y + x[k].z + x[k].w, 0x01010101u, 0u);
        const int row = base + r_off + k * r_step;
        if (warp_row) {
          cnt = __reduce_add_sync(0xffffffffu, cnt);
          if ((tid & 31) == 0 && cnt) atomicAdd(&row_acc[row], cnt);
        } else {
          for (int off = 1; off < cpr; off <<= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
          if (c == 0) row_acc[row] = cnt;  // the lane group holds the whole row
        }
      }
      pending += kStageUnits;
      if (pending + kStageUnits > 255) flush_cols();
    } else if (ok && active) {
      for (int rl = r_off; rl < nr; rl += r_step) {
        uint4 x = *reinterpret_cast<const uint4*>(src + rl * nK);
        if (CAUSAL) x = keep_causal(x, c * 16, row0 + base + rl);
        const uint32_t f0 = nonzero_byte_flags(x.x), f1 = nonzero_byte_flags(x.y);
        const uint32_t f2 = nonzero_byte_flags(x.z), f3 = nonzero_byte_flags(x.w);
        acc[0] += f0; acc[1] += f1; acc[2] += f2; acc[3] += f3;
        int cnt = __popc(f0) + __popc(f1) + __popc(f2) + __popc(f3);
        if (warp_row) {
          cnt = __reduce_add_sync(0xffffffffu, cnt);
          if ((tid & 31) == 0 && cnt) atomicAdd(&row_acc[base + rl], cnt);
        } else if (cnt) {
          atomicAdd(&row_acc[base + rl], cnt);
        }
        if (++pending == 255) flush_cols();
      }
    }
    if (!__syncthreads_and(ok)) {  // every thread has read stage i % kStages, or the CTA gives up
      failed = i;
      break;
    }
    if (tid == 0 && i + kStages < n_chunks) issue(i + kStages);
  }
  if (failed >= 0) {
    if (tid == 0) {
      // let the copies still in flight land before the ring is reused or the CTA exits
      for (int j = failed; j < min(failed + kStages, n_chunks); ++j) {
        const uint32_t bar = smem_u32(&full[j % kStages]);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar, (j / kStages) & 1) && globaltimer() - t0 < kDrainLimitNs) {
        }
      }
    }
    __syncthreads();
  }

  // row loads (exact per CTA) and the CTA's total
  int local = 0;
  for (int r = tid; r < rows; r += kThreads) {
    const int v = row_acc[r];
    row_loads[head * nQ + row0 + r] = v;
    local += v;
  }
  local = __reduce_add_sync(0xffffffffu, local);
  if ((tid & 31) == 0 && local) atomicAdd(&cta_total, local);

  // column partials: each thread's 16 counts go to its own slot of the (now idle) stage
  // ring, [r_off][nK] ints (r_step * nK * 4 <= 16 KB); a thread then sums 4 adjacent
  // columns over the r_step slots and pushes the sums (one 16-byte store) into the
  // shared memory of the rank that owns them (column j belongs to rank j / slice, slice
  // a multiple of 4), at row `rank` of that rank's [n_ranks][slice] receive buffer.
  // Pushing (remote stores) instead of pulling (remote loads) leaves one cluster barrier
  // and no remote round trips.
  int* slot = reinterpret_cast<int*>(stage);
  if (active) {
#pragma unroll
    for (int b = 0; b < 16; b += 4) {
      int4 v;
      v.x = cols[b + 0] + ((acc[b >> 2] >> 0) & 0xff);
      v.y = cols[b + 1] + ((acc[b >> 2] >> 8) & 0xff);
      v.z = cols[b + 2] + ((acc[b >> 2] >> 16) & 0xff);
      v.w = cols[b + 3] + ((acc[b >> 2] >> 24) & 0xff);
      *reinterpret_cast<int4*>(slot + r_off * nK + c * 16 + b) = v;
    }
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid == 0) cluster.map_shared_rank(head_part, 0)[rank] = cta_total;
  const int slice = ((nK + n_ranks - 1) / n_ranks + 3) & ~3;
  for (int j = 4 * tid; j < nK; j += 4 * kThreads) {
    int4 sum = make_int4(0, 0, 0, 0);
    for (int q = 0; q < r_step; ++q) {
      const int4 v = *reinterpret_cast<const int4*>(slot + q * nK + j);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int owner = j / slice;
    *reinterpret_cast<int4*>(cluster.map_shared_rank(recv, owner) + rank * slice + (j - owner * slice)) = sum;
  }
  cluster.sync();  // every rank's pushes have landed

  const int j0 = rank * slice, j1 = min(nK, j0 + slice);
  for (int j = j0 + tid; j < j1; j += kThreads) {
    int sum = 0;
    for (int q = 0; q < n_ranks; ++q) sum += recv[q * slice + (j - j0)];
    col_loads[head * nK + j] = sum;
  }
  if (rank == 0 && tid == 0 && head_loads) {
    int sum = 0;
    for (int q = 0; q < n_ranks; ++q) sum += head_part[q];
    head_loads[head] = sum;
  }
}

// Dense-block lists: for every row r of the mask (B*H*nQ rows of nK blocks), the KV-block
// indices of its dense blocks in ascending order, cols[r * nK + 0 .. counts[r] - 1] (with
// CAUSAL only the blocks on or below the diagonal). A row takes G lanes of a warp (G a power
// of two, 16 G columns per pass: rows of up to 512 blocks in one pass, 32 / G rows per
// warp; longer rows a whole warp, 512 columns at a time): lane l of the row holds 16
// columns as a bit mask, and a prefix sum over the row's lanes gives each lane where its
// indices go.
template <bool VEC, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) dense_lists_kernel(const uint8_t* __restrict__ mask, long long rows,
                                                               int nQ, int nK, int G, int32_t* __restrict__ counts,
                                                               uint16_t* __restrict__ cols) {
  griddep_wait();  // the mask may come from the previous grid
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int sub = lane / G, sl = lane % G;
  const long long r = ((long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * (32 / G) + sub;
  const bool live = r < rows;
  const int limit = !live ? 0 : (CAUSAL ? min(nK, (int)(r % nQ) + 1) : nK);
  const int warp_limit = __reduce_max_sync(0xffffffffu, limit);
  const uint8_t* row = mask + (live ? r : 0) * nK;
  uint16_t* out = cols + (live ? r : 0) * nK;
  int base = 0;
  for (int c0 = 0; c0 < warp_limit; c0 += 16 * G) {
    const int col = c0 + 16 * sl;
    const int rem = limit - col;
    uint32_t bits = 0;
    if (rem > 0) {
      if (VEC) {
        const uint4 x = *reinterpret_cast<const uint4*>(row + col);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) bits |= ((nonzero_byte_flags(w[k]) * 0x01020408u) >> 24) << (4 * k);
      } else {
        for (int t = 0; t < 16 && t < rem; ++t) bits |= (row[col + t] != 0 ? 1u : 0u) << t;
      }
      if (rem < 16) bits &= (1u << rem) - 1u;
    }
    const int cnt = __popc(bits);
    int incl = cnt;
    for (int o = 1; o < G; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o, G);
      if (sl >= o) incl += y;
    }
    int at = base + incl - cnt;
    while (bits) {
      out[at++] = (uint16_t)(col + __ffs(bits) - 1);
      bits &= bits - 1;
    }
    base += __shfl_sync(0xffffffffu, incl, G - 1, G);
  }
  if (live && sl == 0) counts[r] = base;
}

// KV-block loads summed over (b, h): thread j adds column j of every head.
__global__ void __launch_bounds__(kThreads) kv_block_loads_kernel(const int32_t* __restrict__ col_loads,
                                                                  int groups, int nK,
                                                                  int32_t* __restrict__ kv_loads) {
  const int j = blockIdx.x * kThreads + threadIdx.x;
  if (j >= nK) return;
  int s = 0;
  for (int g = 0; g < groups; ++g) s += __ldg(col_loads + (long long)g * nK + j);
  kv_loads[j] = s;
}

// KV-shard masks: thread u takes 16 mask bytes (VEC = 16) or one (VEC = 1) and writes
// them to every shard with the columns of the other shards cleared.
template <int VEC>
__global__ void __launch_bounds__(kThreads) shard_masks_kernel(const uint8_t* __restrict__ mask, long long units,
                                                               int nK, const int32_t* __restrict__ shard_of,
                                                               int n_shards, uint8_t* __restrict__ out, int* err) {
  griddep_wait();  // the mask and the shard plan may come from the previous grids
  griddep_launch_dependents();
  const long long total = units * VEC;  // mask bytes
  const long long stride = (long long)gridDim.x * kThreads;
  for (long long u = (long long)blockIdx.x * kThreads + threadIdx.x; u < units; u += stride) {
    const int col0 = (int)((u * VEC) % nK);
    if constexpr (VEC == 16) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(mask) + u);
      int sh[16];
#pragma unroll
      for (int b = 0; b < 16; ++b) {
        sh[b] = __ldg(shard_of + col0 + b);
        if ((unsigned)sh[b] >= (unsigned)n_shards) dbsp::report(err, DBSP_ERR_INVALID_ARG);
      }
      for (int s = 0; s < n_shards; ++s) {
        uint32_t keep[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t k = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) k |= (sh[4 * w + b] == s ? 0xffu : 0u) << (8 * b);
          keep[w] = k;
        }
        const uint4 y = make_uint4(x.x & keep[0], x.y & keep[1], x.z & keep[2], x.w & keep[3]);
        reinterpret_cast<uint4*>(out + (long long)s * total)[u] = y;
      }
    } else {
      const uint8_t x = __ldg(mask + u);
      const int sh = __ldg(shard_of + col0);
      if ((unsigned)sh >= (unsigned)n_shards) dbsp::report(err, DBSP_ERR_INVALID_ARG);
      for (int s = 0; s < n_shards; ++s) out[(long long)s * total + u] = sh == s ? x : (uint8_t)0;
    }
  }
}

}  // namespace

extern "C" int dbsp_kv_block_loads(const int32_t* col_loads, int groups, int nK, int32_t* kv_loads,
                                   void* stream) {
  if (!col_loads || !kv_loads || groups < 1 || nK < 1) return DBSP_ERR_INVALID_ARG;
  if ((long long)groups * nK >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (!dbsp::aligned(col_loads, 4) || !dbsp::aligned(kv_loads, 4)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  kv_block_loads_kernel<<<(nK + kThreads - 1) / kThreads, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      col_loads, groups, nK, kv_loads);
  DBSP_LAUNCH_CHECK("launch kv_block_loads");
  return DBSP_OK;
}

namespace {

template <bool CAUSAL>
int mask_loads(const uint8_t* mask, int B, int H, int nQ, int nK, int32_t* row_loads, int32_t* col_loads,
               int32_t* head_loads, void* stream) {
  if (!mask || !row_loads || !col_loads) return DBSP_ERR_INVALID_ARG;
  if (CAUSAL && nQ != nK) return DBSP_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || nQ < 1 || nK < 1) return DBSP_ERR_INVALID_ARG;
  const long long total = (long long)B * H * nQ * nK;
  if (total >= (1LL << 31) || (long long)B * H > 65535) return DBSP_ERR_INVALID_ARG;
  if (nK > kMaxCols || nQ > kMaxRows) return DBSP_ERR_UNSUPPORTED;
  if (!dbsp::aligned(row_loads, 4) || !dbsp::aligned(col_loads, 4) ||
      (head_loads && !dbsp::aligned(head_loads, 4)))
    return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;

  // band of rows per CTA: about 16 KB of mask per CTA, at most 8 CTAs per head
  const long long head_bytes = (long long)nQ * nK;
  int ranks = (int)std::min<long long>(kMaxCluster, std::max<long long>(1, (head_bytes + 16383) / 16384));
  ranks = std::min(ranks, nQ);
  const int rows_per_cta = (nQ + ranks - 1) / ranks;
  ranks = (nQ + rows_per_cta - 1) / rows_per_cta;
  const bool vec = (nK % 16 == 0) && dbsp::aligned(mask, 16);
  const size_t part_bytes = sizeof(int) * ((size_t)nK + 4 * kMaxCluster + rows_per_cta);
  const bool stream_rows = vec && nK <= kStreamMaxCols && part_bytes + kStages * kStageBytes <= kStreamMaxSmem;
  const size_t smem = part_bytes + (stream_rows ? (size_t)kStages * kStageBytes : 0);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ranks, B * H, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ranks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = dbsp::overlap_previous_grid();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  if (stream_rows) {
    e = cudaFuncSetAttribute(mask_loads_stream_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(mask_loads)");
    if (kMaxCluster > 8) {
      e = cudaFuncSetAttribute(mask_loads_stream_kernel<CAUSAL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(mask_loads cluster)");
    }
    const int chunk_rows = kStageBytes / nK;
    e = cudaLaunchKernelEx(&cfg, mask_loads_stream_kernel<CAUSAL>, mask, nQ, nK, rows_per_cta, chunk_rows, row_loads,
                           col_loads, head_loads, dbsp::error_word(dev));
    if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch mask_loads");
    return DBSP_OK;
  }
  auto kernel = vec ? mask_loads_kernel<16, CAUSAL> : mask_loads_kernel<1, CAUSAL>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(mask_loads)");
  if (kMaxCluster > 8) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(mask_loads cluster)");
  }
  e = cudaLaunchKernelEx(&cfg, kernel, mask, nQ, nK, rows_per_cta, row_loads, col_loads, head_loads);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch mask_loads");
  return DBSP_OK;
}

int dense_lists(const uint8_t* mask, int B, int H, int nQ, int nK, int causal, int32_t* counts, uint16_t* cols,
                void* stream) {
  if (!mask || !counts || !cols) return DBSP_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || nQ < 1 || nK < 1) return DBSP_ERR_INVALID_ARG;
  if (causal && nQ != nK) return DBSP_ERR_INVALID_ARG;
  if ((long long)B * H * nQ * nK >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (nK > 65536) return DBSP_ERR_UNSUPPORTED;  // indices are 16-bit
  if (!dbsp::aligned(counts, 4) || !dbsp::aligned(cols, 2)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  const long long rows = (long long)B * H * nQ;
  const bool vec = (nK % 16 == 0) && dbsp::aligned(mask, 16);
  int G = 1;  // lanes per row: 16 G columns cover min(nK, 512)
  while (G < 32 && 16 * G < nK) G <<= 1;
  const long long per_cta = (kThreads / 32) * (32 / G);
  const dim3 grid((unsigned)((rows + per_cta - 1) / per_cta));
  cudaError_t e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (vec)
    e = causal ? dbsp::launch_overlapped(dense_lists_kernel<true, true>, grid, dim3(kThreads), 0, s, mask, rows, nQ,
                                         nK, G, counts, cols)
               : dbsp::launch_overlapped(dense_lists_kernel<true, false>, grid, dim3(kThreads), 0, s, mask, rows, nQ,
                                         nK, G, counts, cols);
  else
    e = causal ? dbsp::launch_overlapped(dense_lists_kernel<false, true>, grid, dim3(kThreads), 0, s, mask, rows, nQ,
                                         nK, G, counts, cols)
               : dbsp::launch_overlapped(dense_lists_kernel<false, false>, grid, dim3(kThreads), 0, s, mask, rows, nQ,
                                         nK, G, counts, cols);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch dense_lists");
  return DBSP_OK;
}

}  // namespace

extern "C" int dbsp_dense_block_lists(const uint8_t* mask, int B, int H, int nQ, int nK, int causal,
                                      int32_t* counts, uint16_t* cols, void* stream) {
  return dense_lists(mask, B, H, nQ, nK, causal, counts, cols, stream);
}

extern "C" int dbsp_block_mask_loads(const uint8_t* mask, int B, int H, int nQ, int nK, int32_t* row_loads,
                                     int32_t* col_loads, int32_t* head_loads, void* stream) {
  return mask_loads<false>(mask, B, H, nQ, nK, row_loads, col_loads, head_loads, stream);
}

extern "C" int dbsp_block_mask_loads_causal(const uint8_t* mask, int B, int H, int nQ, int nK,
                                            int32_t* row_loads, int32_t* col_loads, int32_t* head_loads,
                                            void* stream) {
  return mask_loads<true>(mask, B, H, nQ, nK, row_loads, col_loads, head_loads, stream);
}

extern "C" int dbsp_shard_masks(const uint8_t* mask, int B, int H, int nQ, int nK, const int32_t* shard_of,
                                int n_shards, uint8_t* out, void* stream) {
  if (!mask || !shard_of || !out) return DBSP_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || nQ < 1 || nK < 1 || n_shards < 1 || n_shards > 65535) return DBSP_ERR_INVALID_ARG;
  const long long total = (long long)B * H * nQ * nK;
  if (total >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  if (!dbsp::aligned(shard_of, 4)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  const bool vec = nK % 16 == 0 && dbsp::aligned(mask, 16) && dbsp::aligned(out, 16);
  const long long units = vec ? total / 16 : total;
  const int blocks = (int)std::max<long long>(
      1, std::min<long long>((units + kThreads - 1) / kThreads, (long long)dbsp::sm_count(dev) * 8));
  cudaError_t e = vec ? dbsp::launch_overlapped(shard_masks_kernel<16>, dim3(blocks), dim3(kThreads), 0,
                                                static_cast<cudaStream_t>(stream), mask, units, nK, shard_of,
                                                n_shards, out, dbsp::error_word(dev))
                      : dbsp::launch_overlapped(shard_masks_kernel<1>, dim3(blocks), dim3(kThreads), 0,
                                                static_cast<cudaStream_t>(stream), mask, units, nK, shard_of,
                                                n_shards, out, dbsp::error_word(dev));
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch shard_masks");
  return DBSP_OK;
}
