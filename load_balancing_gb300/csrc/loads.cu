// Mask loads: dense-block counts per Q-block row, per KV-block column and per head.
//
// db-SP blog, scenario 2, first bullet: a Q-block's load is the number of dense
// blocks in its mask row, a KV-block's load the number in its column; scenario 1
// balances whole heads, whose load is the head's total.
//
// Design: a thread-block cluster of up to 8 CTAs per (b, h) head. Each CTA scans a
// band of rows with 16-byte vector loads (byte-granular when the row length or
// the pointer does not allow it). Row loads are exact per CTA and written
// directly; column partials live in shared memory and are summed by cluster rank
// 0 through distributed shared memory, so no global scratch or atomics on the
// outputs are needed and the outputs need no prior zeroing. HBM-bound: every mask
// byte is read once.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCluster = 8;
constexpr int kMaxCols = 16384;  // column partials in shared memory: 64 KB

// Number of non-zero bytes in a 32-bit word, as 0x01 flags per byte.
__device__ __forceinline__ uint32_t nonzero_byte_flags(uint32_t x) {
  return ((((x & 0x7f7f7f7fu) + 0x7f7f7f7fu) | x) >> 7) & 0x01010101u;
}

// VEC = 16: each work unit is 16 consecutive mask bytes of one row (uint4 loads);
// VEC = 1: one byte.
template <int VEC>
__global__ void __launch_bounds__(kThreads) mask_loads_kernel(
    const uint8_t* __restrict__ mask, int nQ, int nK, int rows_per_cta,
    int32_t* __restrict__ row_loads, int32_t* __restrict__ col_loads,
    int32_t* __restrict__ head_loads) {
  extern __shared__ int smem[];
  int* col_part = smem;               // [nK]
  int* row_acc = smem + nK;           // [rows_per_cta]
  __shared__ int cta_total;

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
          const int nz = __ldg(head_mask + (long long)r * nK + c) != 0;
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

extern "C" int dbsp_block_mask_loads(const uint8_t* mask, int B, int H, int nQ, int nK,
                                     int32_t* row_loads, int32_t* col_loads,
                                     int32_t* head_loads, void* stream) {
  if (!mask || !row_loads || !col_loads) return DBSP_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || nQ < 1 || nK < 1) return DBSP_ERR_INVALID_ARG;
  const long long total = (long long)B * H * nQ * nK;
  if (total >= (1LL << 31) || (long long)B * H > 65535) return DBSP_ERR_INVALID_ARG;
  if (nK > kMaxCols) return DBSP_ERR_UNSUPPORTED;
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
  const size_t smem = sizeof(int) * ((size_t)nK + rows_per_cta);

  const bool vec = (nK % 16 == 0) && dbsp::aligned(mask, 16);
  auto kernel = vec ? mask_loads_kernel<16> : mask_loads_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(mask_loads)");

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ranks, B * H, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ranks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, mask, nQ, nK, rows_per_cta, row_loads, col_loads, head_loads);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch mask_loads");
  return DBSP_OK;
}
