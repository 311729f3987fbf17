// Merge of (O, m, l) partials from KV shards into the final output.
//
// 6D attention notes §2.1, step 3 of the ring loop and its last line: the running
// maximum is the larger maximum, each side is rescaled by exp(old max - new max),
// row sums and unnormalised outputs add with those weights, and the output is
// divided by the row sum at the end. Folding n shards that way equals the
// one-shot form m* = max_k m_k, w_k = exp(m_k - m*), l = sum w_k l_k,
// O = sum w_k O_k / l, which this kernel evaluates (fewer dependent steps).
// A partial with l_k == 0 or m_k == -inf is empty and contributes nothing.
//
// Layout: o_parts [n_shards, rows, d] fp32, m/l [n_shards, rows] fp32. One thread
// owns four float4 groups of a row, strided so that each load instruction of a warp
// reads contiguous 128-byte runs (streaming cache hint), and writes them as bf16
// (8-byte stores); the shard weights are computed once per thread for its 16 elements. HBM-bound: each live partial is read exactly once.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8;  // shards whose loads are in flight together
constexpr int kQuads = 4;  // float4 groups of one row per thread (16 consecutive elements)

__global__ void __launch_bounds__(kThreads) merge_partials_kernel(
    const float* __restrict__ o_parts, const float* __restrict__ m_parts,
    const float* __restrict__ l_parts, int n_shards, long long rows, int d,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  dbsp::ptx::griddep_wait();  // the partials come from the previous grids
  dbsp::ptx::griddep_launch_dependents();
  const int quads = d >> 2;
  const int groups = (quads + kQuads - 1) / kQuads;  // threads per row
  const long long total = rows * groups;
  const long long stride = (long long)gridDim.x * kThreads;
  for (long long u = (long long)blockIdx.x * kThreads + threadIdx.x; u < total; u += stride) {
    const long long row = u / groups;
    const int qt = (int)(u - row * groups);  // this thread's float4s: qt, qt + groups, ... (coalesced)
    // pass 1: m* over live partials
    float mstar = -INFINITY;
    for (int k = 0; k < n_shards; ++k) {
      const float mk = __ldg(m_parts + (long long)k * rows + row);
      const float lk = __ldg(l_parts + (long long)k * rows + row);
      if (lk > 0.f && mk > -INFINITY) mstar = fmaxf(mstar, mk);
    }
    float4 acc[kQuads];
#pragma unroll
    for (int i = 0; i < kQuads; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (mstar > -INFINITY) {
      // pass 2, kChunk shards at a time: the weights first, then the chunk's partial
      // loads as independent predicated streams (an empty partial is never read),
      // then the weighted sums
      for (int k0 = 0; k0 < n_shards; k0 += kChunk) {
        float w[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          const int k = k0 + j;
          w[j] = 0.f;
          if (k < n_shards) {
            const float mk = __ldg(m_parts + (long long)k * rows + row);
            const float lk = __ldg(l_parts + (long long)k * rows + row);
            if (lk > 0.f && mk > -INFINITY) {
              w[j] = expf(mk - mstar);
              l += w[j] * lk;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          if (w[j] > 0.f) {
            const float4* src = reinterpret_cast<const float4*>(o_parts + ((long long)(k0 + j) * rows + row) * d) + qt;
            float4 o[kQuads];
#pragma unroll
            for (int i = 0; i < kQuads; ++i)
              o[i] = qt + i * groups < quads ? __ldcs(src + i * groups) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kQuads; ++i) {
              acc[i].x += w[j] * o[i].x; acc[i].y += w[j] * o[i].y;
              acc[i].z += w[j] * o[i].z; acc[i].w += w[j] * o[i].w;
            }
          }
        }
      }
      const float inv = 1.f / l;
#pragma unroll
      for (int i = 0; i < kQuads; ++i) { acc[i].x *= inv; acc[i].y *= inv; acc[i].z *= inv; acc[i].w *= inv; }
    }
#pragma unroll
    for (int i = 0; i < kQuads; ++i) {
      if (qt + i * groups < quads) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x, acc[i].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z, acc[i].w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        __stcs(reinterpret_cast<uint2*>(out + row * d) + qt + i * groups, packed);
      }
    }
    if (lse && qt == 0) lse[row] = mstar > -INFINITY ? mstar + logf(l) : -INFINITY;
  }
}

// The pieces of every split item (slots split_off[s] .. split_off[s + 1] - 1, each
// `block` rows of o/m/l) combined into the item's output rows, with the same one-shot
// form as above. One warp per output row, four consecutive columns per lane (d <= 128);
// the number of split items is read from counts[2] on the device, so the grid strides
// over an upper bound.
__global__ void __launch_bounds__(kThreads) merge_pieces_kernel(
    const float* __restrict__ o_piece, const float* __restrict__ m_piece, const float* __restrict__ l_piece,
    const int32_t* __restrict__ split_item, const int32_t* __restrict__ split_off,
    const int32_t* __restrict__ counts, int max_slots, int n_items, int nQ, int S, int block, int d,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int* err) {
  dbsp::ptx::griddep_wait();  // the pieces come from the previous grid
  dbsp::ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int n_split = counts[2];
  const int n_slots = min(counts[3], max_slots);  // slots that hold pieces, within the buffers
  if (n_split < 0 || n_split > n_items) {
    if (blockIdx.x == 0 && threadIdx.x == 0) dbsp::report(err, DBSP_ERR_INVALID_ARG);
    return;
  }
  const long long rows = (long long)n_split * block;
  const long long warps = (long long)gridDim.x * (kThreads / 32);
  for (long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); row < rows; row += warps) {
    const int si = (int)(row / block), r = (int)(row - (long long)si * block);
    const int item = split_item[si], s0 = split_off[si], s1 = split_off[si + 1];
    if (item < 0 || item >= n_items || s0 < 0 || s1 < s0 || s1 > n_slots) {
      if (lane == 0) dbsp::report(err, DBSP_ERR_INVALID_ARG);
      continue;
    }
    const long long grow = (long long)(item / nQ) * S + (long long)(item % nQ) * block + r;
    float mstar = -INFINITY;
    for (int sl = s0; sl < s1; ++sl) {
      const long long pr = (long long)sl * block + r;
      const float mk = __ldg(m_piece + pr), lk = __ldg(l_piece + pr);
      if (lk > 0.f && mk > -INFINITY) mstar = fmaxf(mstar, mk);
    }
    const int c = lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (mstar > -INFINITY) {
      for (int sl = s0; sl < s1; ++sl) {
        const long long pr = (long long)sl * block + r;
        const float mk = __ldg(m_piece + pr), lk = __ldg(l_piece + pr);
        if (!(lk > 0.f && mk > -INFINITY)) continue;  // an empty piece's O is never read
        const float w = expf(mk - mstar);
        l += w * lk;
        if (c < d) {
          const float4 x = __ldcs(reinterpret_cast<const float4*>(o_piece + pr * d + c));
          acc.x += w * x.x;
          acc.y += w * x.y;
          acc.z += w * x.z;
          acc.w += w * x.w;
        }
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (c < d) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&a);
      v.y = *reinterpret_cast<const uint32_t*>(&b);
      *reinterpret_cast<uint2*>(out + grow * d + c) = v;
    }
    if (lse && lane == 0) lse[grow] = l > 0.f ? mstar + logf(l) : -INFINITY;
  }
}

}  // namespace

extern "C" int dbsp_merge_partials(const float* o_parts, const float* m_parts, const float* l_parts,
                                   int n_shards, int64_t rows, int d, void* out, float* lse,
                                   void* stream) {
  if (n_shards < 1 || rows < 0 || d < 4 || d > 1024 || (d % 4) != 0) return DBSP_ERR_INVALID_ARG;
  if (rows == 0) return DBSP_OK;
  if (!o_parts || !m_parts || !l_parts || !out) return DBSP_ERR_INVALID_ARG;
  if (!dbsp::aligned(o_parts, 16) || !dbsp::aligned(out, 8) || !dbsp::aligned(m_parts, 4) ||
      !dbsp::aligned(l_parts, 4) || (lse && !dbsp::aligned(lse, 4)))
    return DBSP_ERR_INVALID_ARG;
  if ((long long)n_shards * rows * d >= (1LL << 62) / 4) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  const long long units = rows * ((d / 4 + kQuads - 1) / kQuads);
  const long long want = (units + kThreads - 1) / kThreads;
  const int blocks = (int)std::min<long long>(want, (long long)dbsp::sm_count(dev) * 8);
  const cudaError_t e = dbsp::launch_overlapped(merge_partials_kernel, dim3(blocks), dim3(kThreads), 0,
                                                static_cast<cudaStream_t>(stream), o_parts, m_parts, l_parts,
                                                n_shards, rows, d, static_cast<__nv_bfloat16*>(out), lse);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch merge_partials");
  return DBSP_OK;
}

extern "C" int dbsp_merge_pieces(const float* o_piece, const float* m_piece, const float* l_piece,
                                 const int32_t* split_item, const int32_t* split_off, const int32_t* counts,
                                 int max_slots, int B, int H, int S, int d, int block, void* out, float* lse,
                                 void* stream) {
  if (B < 1 || H < 1 || S < 1 || (d != 64 && d != 128) || block < 1 || S % block != 0) return DBSP_ERR_INVALID_ARG;
  if (max_slots < 0) return DBSP_ERR_INVALID_ARG;
  if (!o_piece || !m_piece || !l_piece || !split_item || !split_off || !counts || !out) return DBSP_ERR_INVALID_ARG;
  if (!dbsp::aligned(o_piece, 16) || !dbsp::aligned(out, 8) || !dbsp::aligned(m_piece, 4) ||
      !dbsp::aligned(l_piece, 4) || (lse && !dbsp::aligned(lse, 4)))
    return DBSP_ERR_INVALID_ARG;
  const long long n_items = (long long)B * H * (S / block);
  if ((long long)B * H * S >= (1LL << 31)) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  const long long want = (n_items * block + (kThreads / 32) - 1) / (kThreads / 32);
  const int blocks = (int)std::max<long long>(1, std::min<long long>(want, (long long)dbsp::sm_count(dev) * 8));
  const cudaError_t e = dbsp::launch_overlapped(
      merge_pieces_kernel, dim3(blocks), dim3(kThreads), 0, static_cast<cudaStream_t>(stream), o_piece, m_piece,
      l_piece, split_item, split_off, counts, max_slots, (int)n_items, S / block, S, block, d,
      static_cast<__nv_bfloat16*>(out), lse, dbsp::error_word(dev));
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch merge_pieces");
  return DBSP_OK;
}
