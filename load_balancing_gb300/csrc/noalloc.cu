// Split attention (units + piece merge) whose piece scratch is a static device array.
//
// The split path (dbsp_block_sparse_attn_fwd_units, then dbsp_merge_pieces) keeps the
// partial results of the pieces of split items in scratch buffers that the caller
// allocates. Some callers cannot allocate device memory at the point where they run
// attention: code running under an allocator that must not grow or fragment (a serving
// runtime that reserved its memory pool up front), or a host thread that may not call
// cudaMalloc (it would synchronise the device, or it runs inside another library's
// callback). This file gives them one entry point that allocates nothing: the pieces
// live in a file-scope __device__ array of fixed size, which every GPU that loads the
// library holds until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it names a
// host-side stand-in), so the first call on each device, with that device current,
// looks the address up with cudaGetSymbolAddress and caches it.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DBSP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_piece_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch[kMaxDevices];  // device address of g_piece_scratch, per device

// The scratch's device address on `dev` (the current device), looked up once.
int scratch_address(int dev, void** ptr) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_piece_scratch);
    if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaGetSymbolAddress(piece scratch)");
    g_scratch[dev] = p;
  }
  *ptr = g_scratch[dev];
  return DBSP_OK;
}

}  // namespace

extern "C" int dbsp_block_sparse_attn_fwd_split_noalloc(
    const void* q, const void* k, const void* v, const uint8_t* mask, int B, int H, int S, int d, int block,
    int causal, float scale, const int32_t* worker_offsets, const int32_t* worklist, int n_workers,
    const int32_t* unit_item, const int32_t* unit_pk, const int32_t* unit_slot, int n_units,
    const int32_t* split_item, const int32_t* split_off, const int32_t* counts, int max_slots, void* out,
    float* lse, int64_t* cta_timing, void* stream) {
  if (max_slots < 0 || block < 1 || d < 1) return DBSP_ERR_INVALID_ARG;
  // pieces take max_slots * block rows of d fp32 (O) plus 2 fp32 (m, l)
  const unsigned long long need = (unsigned long long)max_slots * (unsigned long long)block *
                                  (unsigned long long)(d + 2) * sizeof(float);
  if (need > kScratchBytes) return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  if (dev >= kMaxDevices) return DBSP_ERR_UNSUPPORTED;
  void* base = nullptr;
  st = scratch_address(dev, &base);
  if (st != DBSP_OK) return st;
  float* o_piece = static_cast<float*>(base);
  float* m_piece = o_piece + (size_t)max_slots * block * d;
  float* l_piece = m_piece + (size_t)max_slots * block;
  st = dbsp_block_sparse_attn_fwd_units(q, k, v, mask, B, H, S, d, block, causal, scale, worker_offsets, worklist,
                                        n_workers, unit_item, unit_pk, unit_slot, n_units, out, lse, o_piece,
                                        m_piece, l_piece, max_slots, cta_timing, stream);
  if (st != DBSP_OK) return st;
  return dbsp_merge_pieces(o_piece, m_piece, l_piece, split_item, split_off, counts, max_slots, B, H, S, d, block,
                           out, lse, stream);
}
