// Block-sparse attention forward over an LPT worklist, for sm_103a.
//
// What is computed (6D attention notes §2.1, step 2 and the final division; db-SP
// blog, scenario 2): for every item (b, h, qb) the query rows of Q-block qb attend
// to the keys of the dense KV-blocks of mask row (b, h, qb); the result is the
// online-softmax accumulation O / l with LSE = m + ln l, or the unnormalised
// partial (O, m, l) of one KV shard. Causal (6D attention notes §2.3): blocks
// above the diagonal are skipped and the diagonal block is masked per element.
//
// Design: one persistent CTA per worker walking its worklist; dense blocks are
// numbered G = 0, 1, ... across the worker's items. TMEM holds the O accumulator and
// THREE S buffers (O | S0 | S1 | S2), and P(G) is written over the first block/2
// columns of its own S buffer, so S(G+1) and S(G+2) run on the tensor core while
// the softmax of block G works, and the next P never waits for the previous PV.
// 12 warps:
//   warp 0      producer of Q and K: reads each item's mask row 16 bytes per lane,
//               publishes (id, dense count), TMA-loads the Q tile (two buffers) and
//               the dense K tiles into a ring; an item without dense blocks is not
//               published: this warp writes its output rows itself;
//   warp 1      producer of V: walks the same items and loads the dense V tiles into
//               a second ring (S runs ahead of PV, so K and V are consumed at
//               different times);
//   warp 2      TMEM owner; lane 0 issues S(G) = Q K_G^T (tcgen05.mma M=128
//               N=block K=d, both operands in shared memory) into buffer G mod 3,
//               once PV(G-3) has completed;
//   warp 3      lane 0 issues O += P(G) V_G (M=128 N=d K=block, P from TMEM, V from
//               shared memory, MN-major) once the softmax has stored P(G);
//   warps 4..11 softmax: warp 4 + 4 s + q owns the 16 query rows q*32 + s*16 + [0, 16)
//               (TMEM lanes of quarter q). A row is split over two threads of one warp
//               (split 16-lane tcgen05 shape): one holds S columns [0, block/2) and O
//               columns [0, d/2), the other the second halves, so the row maximum and
//               the row sum take one shuffle and no warp waits on another. Diagonal
//               masking; running maximum in base-2 units; P = exp2(S*scale*log2e - m)
//               rounded to bf16 pairs and stored into TMEM with tcgen05.st. O is
//               rescaled in TMEM only when a row's maximum grows by more than 2^8
//               (exact either way: O and l always share one reference maximum), after
//               waiting for the previous PV. Epilogue: O / l and LSE, or the partial
//               triple with the true row maximum.
//
// Every mbarrier wait is bounded (2 s of %globaltimer). On expiry the CTA sets the
// device error word to DBSP_ERR_TIMEOUT, every role leaves its loop, in-flight
// copies and MMAs are waited for (bounded) and TMEM is freed before returning.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace {

using namespace dbsp::ptx;

constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;    // warpgroup 0: 2 producers, 2 MMA issuers; 2 softmax warpgroups
constexpr int kMmaWarp = 2;
constexpr int kSoftmaxWarp0 = 4;
// Register split per SM sub-partition (one warp of each warpgroup): the launch gives
// every warp 168 registers (65536 / 384, rounded down to 8); warpgroup 0 gives back
// down to 104 and each softmax warpgroup grows to 200 (104 + 200 + 200 = 3 x 168).
constexpr uint32_t kRegsControl = 104;
constexpr uint32_t kRegsSoftmax = 200;
static_assert(kRegsControl + 2 * kRegsSoftmax <= 3 * 168, "register split exceeds the launch budget");
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                // S buffers at TMEM columns 128, 256, 384
constexpr uint32_t kSCol = 128;
constexpr int kQBufs = 2;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
// a ring stage is reused after the S (K) or PV (V) that read it completed, tested on the
// per-S-buffer barriers: a ring may not be deeper than the S buffers
static_assert(kKStages <= kSBufs && kVStages <= kSBufs, "ring deeper than the S buffers");
#ifdef DBSP_WAIT_TEST
// Test build only (never the product library): waits give up after 20 ms, and the V
// producer of CTA 0 leaves out its first tile (no arrival, no copy), so that the PV
// issuer's wait for that tile runs out and the whole teardown path runs.
constexpr uint64_t kWaitLimitNs = 20000000ull;      // 20 ms per wait
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s per wait
#endif
constexpr uint64_t kDrainLimitNs = 100000000ull;    // 100 ms per teardown wait
constexpr float kRescaleThreshold = 8.0f;           // log2 units: P <= 256 between rescales

struct AttnParams {
  const uint8_t* mask;
  int H, S, nQ, nK, n_items;
  int causal;
  float scale_log2;
  const int32_t* offsets;
  const int32_t* worklist;
  __nv_bfloat16* out;
  float* lse;
  float* o_part;
  float* m_part;
  float* l_part;
  int64_t* timing;
  int* err;
  // units (optional): worklist entries index a unit table; unit u is piece
  // j = unit_pk[u] & 0xffff of k = unit_pk[u] >> 16 of item unit_item[u], written as a
  // partial to slot unit_slot[u] (k > 1) or as the item's output (k = 1)
  const int32_t* unit_item;
  const int32_t* unit_pk;
  const int32_t* unit_slot;
  int n_units;
  int max_slots;  // capacity of the piece buffers, in slots
  float* o_piece;
  float* m_piece;
  float* l_piece;
  // dense-block lists (optional): row r's dense KV blocks within the causal limit are
  // dense_cols[r * nK + 0 .. dense_n[r] - 1], ascending
  const int32_t* dense_n;
  const uint16_t* dense_cols;
};

template <int BLOCK, int D>
struct Cfg {
  static constexpr int kChunk128 = 128 * 128;             // 128 rows x 128 B (one 64-column chunk)
  static constexpr int kQBytes = (D / 64) * kChunk128;
  static constexpr int kTileChunk = BLOCK * 128;          // BLOCK rows x 128 B
  static constexpr int kTileBytes = (D / 64) * kTileChunk;
  static constexpr int kTx = BLOCK * D * 2;               // bytes of one Q / K / V tile load
  static constexpr int kKOff = kQBufs * kQBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kDataBytes = kVOff + kVStages * kTileBytes;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, BLOCK, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
  static_assert(D <= 128 && BLOCK <= 128, "shape");
};

struct alignas(8) Ctrl {
  uint64_t q_full[kQBufs], q_empty[kQBufs];
  uint64_t k_full[kKStages];
  uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];
  uint64_t epi_full[kQBufs];  // final mode: the 8 softmax warps wrote an item's bf16 output tile
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item_id[2], item_n[2], item_diag[2], item_slot[2];
  alignas(4) uint16_t scan_bits[2][32];  // producers: dense bits of one 512-column mask chunk
  uint32_t tmem_base;
  volatile int abort_flag;
  long long blocks_done;
};

template <int BLOCK, int D>
constexpr size_t smem_bytes() {
  return 1024 + Cfg<BLOCK, D>::kDataBytes + sizeof(Ctrl);
}

// Bounded wait. Returns false on timeout or when another role has aborted.
__device__ __forceinline__ bool wait_bar(Ctrl* c, uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (c->abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        c->abort_flag = 1;
        dbsp::report(err, DBSP_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait taken by every lane of a warp; the warp agrees on the outcome, so that a
// lane that saw the phase complete never runs ahead of one that saw the abort flag
// into a warp-collective instruction.
__device__ __forceinline__ bool warp_wait_bar(Ctrl* c, uint32_t bar, uint32_t parity, int* err) {
  return __all_sync(0xffffffffu, wait_bar(c, bar, parity, err));
}

// Teardown wait: ignores the abort flag, short limit, no error on success.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kDrainLimitNs) break;
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ producers
// 4-bit mask of the non-zero bytes of x (bit i <-> byte i).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t x) {
  const uint32_t t = __vcmpne4(x, 0u) & 0x01010101u;
  return (t * 0x01020408u) >> 24;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

// The mask row of an item is read 512 columns at a time: lane l holds the 16 bytes
// of columns [c0 + 16 l, c0 + 16 l + 16). Rows are read with one 16-byte load per
// lane when every row starts on a 16-byte boundary, else byte by byte.
struct RowScan {
  const uint8_t* mask;
  int nK, nQ, causal;
  bool vec;
  int lane;

  __device__ int limit(int item) const {
    return causal ? min(nK, item % nQ + 1) : nK;
  }
  // dense-block bits of the lane's 16 columns of chunk c0, limited to col < lim
  __device__ uint32_t bits(int item, int c0, int lim) const {
    const int col = c0 + 16 * lane;
    const int rem = lim - col;
    if (rem <= 0) return 0u;
    const uint8_t* row = mask + (long long)item * nK;
    uint32_t b = 0;
    if (vec) {  // col + 16 <= nK: nK is a multiple of 16
      const uint4 v = ld_nc_v4(row + col);
      b = nonzero_bytes(v.x) | (nonzero_bytes(v.y) << 4) | (nonzero_bytes(v.z) << 8) |
          (nonzero_bytes(v.w) << 12);
    } else {
      for (int t = 0; t < 16 && t < rem; ++t) b |= (row[col + t] != 0 ? 1u : 0u) << t;
    }
    return rem < 16 ? b & ((1u << rem) - 1u) : b;
  }
};

// Producer warp `which` (0: Q and K, 1: V). Both walk the worker's items in list
// order; producer 0 also publishes every item to the MMA issuer and the softmax
// warps. `each(col)` is called by lane 0 for the dense blocks of the row, in order.
template <int BLOCK, int D, bool UNITS>
__device__ void run_producer(int which, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                             const AttnParams& p, Ctrl* c, uint8_t* data) {
  using C = Cfg<BLOCK, D>;
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  RowScan rs;
  rs.mask = p.mask;
  rs.nK = p.nK;
  rs.nQ = p.nQ;
  rs.causal = p.causal;
  rs.vec = ((reinterpret_cast<uintptr_t>(p.mask) | (uintptr_t)p.nK) & 15u) == 0;
  rs.lane = lane;
  int begin = p.offsets[blockIdx.x], end = p.offsets[blockIdx.x + 1];
  if (begin < 0 || end < begin) {
    if (lane == 0 && which == 0) dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
    begin = end = 0;
  }
  uint32_t item_cnt = 0, q_cnt = 0, t_cnt = 0;  // items published, Q tiles, K or V tiles (= blocks) issued
  const uint32_t kstages = which == 0 ? kKStages : kVStages;
  // A stage is free once the product that read its previous tile has completed: S for
  // K (s_full), PV for V (pv_done). K lands on k_full; V lands on p_full of its block,
  // next to the softmax warps' arrivals, so the PV issuer tests a single barrier.
  uint64_t* done = which == 0 ? c->s_full : c->pv_done;
  const uint32_t ring = smem_u32(data + (which == 0 ? C::kKOff : C::kVOff));
  const CUtensorMap* map = which == 0 ? tk : tv;
  bool ok = true;
  for (int idx = begin; idx <= end && ok; ++idx) {
    int item = -1, pj = 0, pk = 1, pslot = -1;
    if (idx < end) {
      const int u = __ldg(p.worklist + idx);
      bool valid;
      if constexpr (UNITS) {
        valid = u >= 0 && u < p.n_units;
        if (valid) {
          item = __ldg(p.unit_item + u);
          const int pkw = __ldg(p.unit_pk + u);
          pj = pkw & 0xffff;
          pk = pkw >> 16;
          pslot = __ldg(p.unit_slot + u);
          valid = item >= 0 && item < p.n_items && pk >= 1 && pj < pk &&
                  (pk == 1 ? pslot < 0 : (pslot >= 0 && pslot < p.max_slots));
        }
      } else {
        item = u;
        valid = item >= 0 && item < p.n_items;
      }
      if (!valid) {
        if (lane == 0 && which == 0) dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
        continue;
      }
    }
    // dense blocks of the row within the causal limit: L in all; this unit takes the
    // dense ranks [lo, hi) (piece j of k: floor(j L / k) .. floor((j + 1) L / k))
    int n = 0, limit = 0, lo = 0, hi = INT_MAX;
    long long kv_row0 = 0;
    if (item >= 0) {
      kv_row0 = (long long)(item / p.nQ) * p.S;
      limit = rs.limit(item);
      if (which == 0 || (UNITS && pk > 1)) {
        int L = 0;
        for (int c0 = 0; c0 < limit; c0 += 512) L += __reduce_add_sync(kAll, __popc(rs.bits(item, c0, limit)));
        lo = (int)(((long long)pj * L) / pk);
        hi = (int)(((long long)(pj + 1) * L) / pk);
        n = hi - lo;
      }
    }
    if (which == 0 && item >= 0 && n == 0) {
      // A unit without dense blocks never reaches the MMA issuers or the softmax: this
      // warp writes its rows itself (a piece or partial mode: m = -inf, l = 0, O rows
      // untouched; final mode: O = 0, LSE = -inf).
      const long long row0 = (long long)(item / p.nQ) * p.S + (long long)(item % p.nQ) * BLOCK;
      if (UNITS && pslot >= 0) {
        for (int r = lane; r < BLOCK; r += 32) {
          p.m_piece[(long long)pslot * BLOCK + r] = -INFINITY;
          p.l_piece[(long long)pslot * BLOCK + r] = 0.f;
        }
      } else if (p.o_part) {
        for (int r = lane; r < BLOCK; r += 32) {
          p.m_part[row0 + r] = -INFINITY;
          p.l_part[row0 + r] = 0.f;
        }
      } else {
        uint4* o = reinterpret_cast<uint4*>(p.out + row0 * D);
        for (int i = lane; i < BLOCK * D / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse)
          for (int r = lane; r < BLOCK; r += 32) p.lse[row0 + r] = -INFINITY;
      }
      continue;
    }
    if (which == 0) {  // publish the item
      // the causal diagonal block is the row's last dense block: only the unit ending
      // there masks it
      const int diag = item >= 0 && p.causal && pj == pk - 1 && p.mask[(long long)item * p.nK + item % p.nQ] != 0;
      const uint32_t slot = item_cnt & 1, su = item_cnt >> 1;
      if (lane == 0) {
        ok = wait_bar(c, smem_u32(&c->item_empty[slot]), (su & 1) ^ 1, p.err);
        if (ok) {
          c->item_id[slot] = item;
          c->item_n[slot] = n;
          c->item_diag[slot] = diag;
          c->item_slot[slot] = pslot;
          mbar_arrive(smem_u32(&c->item_full[slot]));
        }
      }
      ok = __shfl_sync(kAll, ok, 0);
      ++item_cnt;
      if (!ok || item < 0) break;
      if (n == 0) continue;
      if (lane == 0) {  // the Q tile of this item
        const uint32_t qs = q_cnt % kQBufs, qu = q_cnt / kQBufs;
        ok = wait_bar(c, smem_u32(&c->q_empty[qs]), (qu & 1) ^ 1, p.err);
        if (ok) {
          const uint32_t qf = smem_u32(&c->q_full[qs]);
          mbar_arrive_expect_tx(qf, C::kTx);
          const int qrow = (int)(kv_row0 + (long long)(item % p.nQ) * BLOCK);
          const uint32_t dst = smem_u32(data) + qs * C::kQBytes;
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch) tma_load_2d(dst + ch * C::kChunk128, tq, ch * 64, qrow, qf);
        }
        ++q_cnt;
      }
      ok = __shfl_sync(kAll, ok, 0);
      if (!ok) break;
    } else if (item < 0) {
      break;
    }
    // the dense K (or V) tiles of the unit, in block order
    int rank = 0;  // dense rank of the next block of the row (lane 0)
    bool past = false;
    for (int c0 = 0; c0 < limit && ok && !past; c0 += 512) {
      c->scan_bits[which][lane] = (uint16_t)rs.bits(item, c0, limit);
      __syncwarp();
      if (lane == 0) {
        const uint32_t* words = reinterpret_cast<const uint32_t*>(c->scan_bits[which]);
        for (int w = 0; w < 16 && ok && !past; ++w) {
          uint32_t wb = words[w];  // columns c0 + 32 w + [0, 32)
          while (wb && ok) {
            const int col = c0 + 32 * w + (__ffs(wb) - 1);
            wb &= wb - 1;
            if constexpr (UNITS) {  // only the unit's dense ranks [lo, hi)
              const int rk = rank++;
              if (rk < lo) continue;
              if (rk >= hi) {
                past = true;
                break;
              }
            }
            const uint32_t s = t_cnt % kstages;
            if (t_cnt >= kstages) {
              const uint32_t prev = t_cnt - kstages;
              ok = wait_bar(c, smem_u32(&done[prev % kSBufs]), (prev / kSBufs) & 1, p.err);
            }
#ifdef DBSP_WAIT_TEST
            if (ok && which == 1 && blockIdx.x == 0 && t_cnt == 0) {  // the left-out tile
              ++t_cnt;
              continue;
            }
#endif
            if (ok) {
              const uint32_t f = smem_u32(which == 0 ? &c->k_full[s] : &c->p_full[t_cnt % kSBufs]);
              mbar_arrive_expect_tx(f, C::kTx);
              const uint32_t dst = ring + s * C::kTileBytes;
              const int row = (int)(kv_row0 + (long long)col * BLOCK);
#pragma unroll
              for (int ch = 0; ch < D / 64; ++ch) tma_load_2d(dst + ch * C::kTileChunk, map, ch * 64, row, f);
              ++t_cnt;
            }
          }
        }
      }
      ok = __shfl_sync(kAll, ok, 0);
      if constexpr (UNITS) past = __shfl_sync(kAll, past, 0);
      __syncwarp();
    }
  }
  // teardown: let every copy this warp started land before shared memory goes away
  if (lane == 0) {
    for (uint32_t k = t_cnt > kstages ? t_cnt - kstages : 0; k < t_cnt; ++k) {
      if (which == 0) drain_bar(smem_u32(&c->k_full[k % kstages]), (k / kstages) & 1);
      else drain_bar(smem_u32(&c->p_full[k % kSBufs]), (k / kSBufs) & 1);
    }
    for (uint32_t k = q_cnt > (uint32_t)kQBufs ? q_cnt - kQBufs : 0; k < q_cnt; ++k)
      drain_bar(smem_u32(&c->q_full[k % kQBufs]), (k / kQBufs) & 1);
  }
  __syncwarp();
}

// Producer warp `which` over precomputed dense-block lists: the schedule of run_producer,
// but an item's dense count and columns are read from the lists instead of its mask row,
// and the next item's worklist entry, count and first 32 columns load while the current
// item's tiles go out. A count outside [0, limit] or a column at or past the limit sets
// DBSP_ERR_INVALID_ARG; the row is then treated as empty, or the tile as block 0, so that
// both producers and the MMA issuers stay in step.
template <int BLOCK, int D>
__device__ void run_producer_listed(int which, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                    const AttnParams& p, Ctrl* c, uint8_t* data) {
  using C = Cfg<BLOCK, D>;
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int nK = p.nK;
  int begin = p.offsets[blockIdx.x], end = p.offsets[blockIdx.x + 1];
  if (begin < 0 || end < begin) {
    if (lane == 0 && which == 0) dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
    begin = end = 0;
  }
  uint32_t item_cnt = 0, q_cnt = 0, t_cnt = 0;
  const uint32_t kstages = which == 0 ? kKStages : kVStages;
  uint64_t* done = which == 0 ? c->s_full : c->pv_done;
  const uint32_t ring = smem_u32(data + (which == 0 ? C::kKOff : C::kVOff));
  const CUtensorMap* map = which == 0 ? tk : tv;
  auto valid_item = [&](int u) { return u >= 0 && u < p.n_items; };
  auto list = [&](int u) { return p.dense_cols + (long long)u * nK; };
  int u_cur = begin < end ? __ldg(p.worklist + begin) : -1;
  int u_nxt = begin + 1 < end ? __ldg(p.worklist + begin + 1) : -1;
  int n_cur = 0;
  uint32_t c_cur = 0;
  if (valid_item(u_cur)) {
    n_cur = __ldg(p.dense_n + u_cur);
    c_cur = lane < nK ? __ldg(list(u_cur) + lane) : 0u;
  }
  bool ok = true;
  for (int idx = begin; idx <= end && ok; ++idx) {
    const int u = u_cur;
    const int n_in = n_cur;
    const uint32_t cw0 = c_cur;
    // the next entry's count and first columns, and the entry after it (used next time)
    int n_nx = 0;
    uint32_t c_nx = 0u;
    if (valid_item(u_nxt)) {
      n_nx = __ldg(p.dense_n + u_nxt);
      c_nx = lane < nK ? __ldg(list(u_nxt) + lane) : 0u;
    }
    const int u_nx2 = idx + 2 < end ? __ldg(p.worklist + idx + 2) : -1;
    u_cur = u_nxt;
    n_cur = n_nx;
    c_cur = c_nx;
    u_nxt = u_nx2;

    int item = -1;
    if (idx < end) {
      item = u;
      if (!valid_item(item)) {
        if (lane == 0 && which == 0) dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
        continue;
      }
    }
    int n = 0, limit = 0;
    long long kv_row0 = 0;
    if (item >= 0) {
      kv_row0 = (long long)(item / p.nQ) * p.S;
      limit = p.causal ? min(nK, item % p.nQ + 1) : nK;
      n = n_in;
      if (n < 0 || n > limit) {
        if (lane == 0 && which == 0) dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
        n = 0;
      }
    }
    if (which == 0 && item >= 0 && n == 0) {
      // an item without dense blocks never reaches the MMA issuers or the softmax: this
      // warp writes its rows itself (partial mode: m = -inf, l = 0; final: O = 0, LSE = -inf)
      const long long row0 = (long long)(item / p.nQ) * p.S + (long long)(item % p.nQ) * BLOCK;
      if (p.o_part) {
        for (int r = lane; r < BLOCK; r += 32) {
          p.m_part[row0 + r] = -INFINITY;
          p.l_part[row0 + r] = 0.f;
        }
      } else {
        uint4* o = reinterpret_cast<uint4*>(p.out + row0 * D);
        for (int i = lane; i < BLOCK * D / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse)
          for (int r = lane; r < BLOCK; r += 32) p.lse[row0 + r] = -INFINITY;
      }
      continue;
    }
    if (which == 0) {  // publish the item
      int diag = 0;
      if (item >= 0 && p.causal) {  // the row's last dense block is the diagonal one
        const int last = n <= 32 ? __shfl_sync(kAll, (int)cw0, n - 1) : (int)__ldg(list(item) + n - 1);
        diag = last == item % p.nQ;
      }
      const uint32_t slot = item_cnt & 1, su = item_cnt >> 1;
      if (lane == 0) {
        ok = wait_bar(c, smem_u32(&c->item_empty[slot]), (su & 1) ^ 1, p.err);
        if (ok) {
          c->item_id[slot] = item;
          c->item_n[slot] = n;
          c->item_diag[slot] = diag;
          c->item_slot[slot] = -1;
          mbar_arrive(smem_u32(&c->item_full[slot]));
        }
      }
      ok = __shfl_sync(kAll, ok, 0);
      ++item_cnt;
      if (!ok || item < 0) break;
      if (lane == 0) {  // the Q tile of this item
        const uint32_t qs = q_cnt % kQBufs, qu = q_cnt / kQBufs;
        ok = wait_bar(c, smem_u32(&c->q_empty[qs]), (qu & 1) ^ 1, p.err);
        if (ok) {
          const uint32_t qf = smem_u32(&c->q_full[qs]);
          mbar_arrive_expect_tx(qf, C::kTx);
          const int qrow = (int)(kv_row0 + (long long)(item % p.nQ) * BLOCK);
          const uint32_t dst = smem_u32(data) + qs * C::kQBytes;
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch) tma_load_2d(dst + ch * C::kChunk128, tq, ch * 64, qrow, qf);
        }
        ++q_cnt;
      }
      ok = __shfl_sync(kAll, ok, 0);
      if (!ok) break;
    } else if (item < 0) {
      break;
    }
    // the dense K (or V) tiles of the item, in block order, 32 columns at a time
    for (int k0 = 0; k0 < n && ok; k0 += 32) {
      const uint32_t cw = k0 == 0 ? cw0 : (k0 + lane < n ? (uint32_t)__ldg(list(item) + k0 + lane) : 0u);
      c->scan_bits[which][lane] = (uint16_t)cw;
      __syncwarp();
      if (lane == 0) {
        const int cnt = min(32, n - k0);
        for (int t = 0; t < cnt && ok; ++t) {
          int col = c->scan_bits[which][t];
          if (col >= limit) {
            dbsp::report(p.err, DBSP_ERR_INVALID_ARG);
            col = 0;
          }
          const uint32_t s = t_cnt % kstages;
          if (t_cnt >= kstages) {
            const uint32_t prev = t_cnt - kstages;
            ok = wait_bar(c, smem_u32(&done[prev % kSBufs]), (prev / kSBufs) & 1, p.err);
          }
#ifdef DBSP_WAIT_TEST
          if (ok && which == 1 && blockIdx.x == 0 && t_cnt == 0) {  // the left-out tile
            ++t_cnt;
            continue;
          }
#endif
          if (ok) {
            const uint32_t f = smem_u32(which == 0 ? &c->k_full[s] : &c->p_full[t_cnt % kSBufs]);
            mbar_arrive_expect_tx(f, C::kTx);
            const uint32_t dst = ring + s * C::kTileBytes;
            const int row = (int)(kv_row0 + (long long)col * BLOCK);
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) tma_load_2d(dst + ch * C::kTileChunk, map, ch * 64, row, f);
            ++t_cnt;
          }
        }
      }
      ok = __shfl_sync(kAll, ok, 0);
      __syncwarp();
    }
  }
  // teardown: let every copy this warp started land before shared memory goes away
  if (lane == 0) {
    for (uint32_t k = t_cnt > kstages ? t_cnt - kstages : 0; k < t_cnt; ++k) {
      if (which == 0) drain_bar(smem_u32(&c->k_full[k % kstages]), (k / kstages) & 1);
      else drain_bar(smem_u32(&c->p_full[k % kSBufs]), (k / kSBufs) & 1);
    }
    for (uint32_t k = q_cnt > (uint32_t)kQBufs ? q_cnt - kQBufs : 0; k < q_cnt; ++k)
      drain_bar(smem_u32(&c->q_full[k % kQBufs]), (k / kQBufs) & 1);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuers
// Two threads issue tcgen05.mma: one the S products, one the PV products. An MMA
// issue holds its thread for about the MMA's duration, so every mbarrier test or
// commit of a single issuer would leave the tensor core idle; with two issuers one
// thread's synchronisation overlaps the other's MMAs. tcgen05.commit tracks the MMAs
// of the committing thread, which is all each barrier below needs.

// S(G) = Q K_G^T into S buffer G mod 3, once PV(G-3) has released that buffer.
template <int BLOCK, int D>
__device__ void run_mma_s(const AttnParams& p, Ctrl* c, uint32_t data, uint32_t tmem) {
  using C = Cfg<BLOCK, D>;
  uint32_t items = 0, G = 0, ks = 0, qc = 0;
  bool ok = true;
  while (ok) {
    const uint32_t slot = items & 1;
    if (!wait_bar(c, smem_u32(&c->item_full[slot]), (items >> 1) & 1, p.err)) break;
    const int item = c->item_id[slot], n = c->item_n[slot];
    mbar_arrive(smem_u32(&c->item_empty[slot]));  // every reader of the slot releases it
    ++items;
    if (item < 0) break;
    if (n == 0) continue;
    const uint32_t qs = qc % kQBufs;
    if (!wait_bar(c, smem_u32(&c->q_full[qs]), (qc / kQBufs) & 1, p.err)) break;
    const uint32_t qa = data + qs * C::kQBytes;
    for (int j = 0; j < n && ok; ++j, ++G, ++ks) {
      const uint32_t b = G % kSBufs, kst = ks % kKStages;
      ok = (G < (uint32_t)kSBufs || wait_bar(c, smem_u32(&c->pv_done[b]), ((G / kSBufs) - 1) & 1, p.err)) &&
           wait_bar(c, smem_u32(&c->k_full[kst]), (ks / kKStages) & 1, p.err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t kb = data + C::kKOff + kst * C::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a = smem_desc_sw128(qa + (kk >> 2) * C::kChunk128 + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * C::kTileChunk + (kk & 3) * 32, 16, 1024);
        mma_bf16_ss(tmem + kSCol + b * 128, a, bd, C::kIdescS, kk > 0);
      }
      mma_commit(smem_u32(&c->s_full[b]));
    }
    if (!ok) break;
    mma_commit(smem_u32(&c->q_empty[qs]));
    ++qc;
  }
  // teardown: every MMA issued by this thread must finish before TMEM is freed
  mma_commit(smem_u32(&c->drain));
}

// O (+)= P(G) V_G once the softmax has stored P(G); releases the item slots.
template <int BLOCK, int D>
__device__ void run_mma_pv(const AttnParams& p, Ctrl* c, uint32_t data, uint32_t tmem) {
  using C = Cfg<BLOCK, D>;
  uint32_t items = 0, G = 0, vs = 0;
  long long blocks = 0;
  bool ok = true;
  while (ok) {
    const uint32_t slot = items & 1;
    if (!wait_bar(c, smem_u32(&c->item_full[slot]), (items >> 1) & 1, p.err)) break;
    const int item = c->item_id[slot], n = c->item_n[slot];
    mbar_arrive(smem_u32(&c->item_empty[slot]));
    ++items;
    if (item < 0) break;
    for (int j = 0; j < n && ok; ++j, ++G, ++vs) {
      const uint32_t b = G % kSBufs, vst = vs % kVStages;
      ok = wait_bar(c, smem_u32(&c->p_full[b]), (G / kSBufs) & 1, p.err);  // P(G) and V(G)
      if (!ok) break;
      tc_fence_after();
      const uint32_t vb = data + C::kVOff + vst * C::kTileBytes;
      const uint32_t pcol = tmem + kSCol + b * 128;
#pragma unroll
      for (int kk = 0; kk < BLOCK / 16; ++kk) {
        const uint64_t bd = smem_desc_sw128(vb + kk * 16 * 128, C::kTileChunk, 1024);
        mma_bf16_ts(tmem, pcol + kk * 8, bd, C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(&c->pv_done[b]));
      ++blocks;
    }
  }
  mma_commit(smem_u32(&c->drain));
  c->blocks_done = blocks;
}

// ------------------------------------------------------------------ softmax + epilogue
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// (a0, a1) * (b, b) + (c, c) as one packed fp32x2 FMA
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Softmax warps: warp 4 + 4 * sub + quarter owns the 16 rows quarter * 32 + sub * 16 + [0, 16)
// of the tile (TMEM lanes of its quarter). Each row is split over two threads of the same
// warp (split 16-lane TMEM shape): thread t < 16 holds columns [0, BLOCK/2) of S and
// [0, D/2) of O for row t, thread t + 16 the other halves. Row maxima and row sums are
// combined with one shuffle, so the softmax warps never wait on one another.
#ifndef DBSP_DEFER_RELEASE
#define DBSP_DEFER_RELEASE 1
#endif
constexpr int kDeferRelease = DBSP_DEFER_RELEASE;  // blocks of P stored before a Q buffer's release

template <int BLOCK, int D, bool UNITS>
__device__ void run_softmax(const AttnParams& p, Ctrl* c, uint32_t tmem, uint32_t data, const CUtensorMap* to) {
  using C = Cfg<BLOCK, D>;
  constexpr int CW = BLOCK / 2;  // S columns per thread
  constexpr int DW = D / 2;      // O columns per thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int sub = (warp - kSoftmaxWarp0) >> 2;
  const int ch = lane >> 4;                          // column half of this thread
  const int r = quarter * 32 + sub * 16 + (lane & 15);  // query row within the tile = TMEM lane
  const bool row_ok = BLOCK == 128 || r < BLOCK;  // a 64-row tile leaves TMEM lanes 64..127 unused
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32 + sub * 16) << 16);
  const bool partial = p.o_part != nullptr;
  const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
  uint32_t items = 0, G = 0;
  // An output tile's TMA store reads its Q buffer for a while after issue; the releaser
  // waits for that read, and releases the buffer, only after it has stored the P of the
  // next kDeferRelease blocks (or at its next epilogue), so that the wait does not hold
  // back the next item's first PV. Lane 0 of the releaser warp, which issued the store.
  int pend_qs = -1, pend_left = 0;
  auto release_pending = [&]() {
    bulk_wait_read_all();
    mbar_arrive(smem_u32(&c->q_empty[pend_qs]));
    pend_qs = -1;
  };
  bool ok = true;
  while (ok) {
    const uint32_t slot = items & 1;
    if (!warp_wait_bar(c, smem_u32(&c->item_full[slot]), (items >> 1) & 1, p.err)) break;
    const int item = c->item_id[slot], n = c->item_n[slot], diag = c->item_diag[slot];
    const int pslot = UNITS ? c->item_slot[slot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&c->item_empty[slot]));
    ++items;
    if (item < 0) break;
    const long long bh = item / p.nQ;
    const int qb = item % p.nQ;
    const long long grow = bh * p.S + (long long)qb * BLOCK + r;  // global query row
    if (n == 0) continue;  // empty items are written by the producer and never published
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j, ++G) {
      const uint32_t b = G % kSBufs, bu = G / kSBufs;
      const uint32_t sbase = lane_base + kSCol + b * 128;
      if (!warp_wait_bar(c, smem_u32(&c->s_full[b]), bu & 1, p.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[CW];
      if constexpr (CW == 64) tmem_ld64s_wait<CW>(sbase, sr);
      else tmem_ld32s_wait<CW>(sbase, sr);
      float* s = reinterpret_cast<float*>(sr);
      if (diag && j == n - 1) {
#pragma unroll
        for (int k = 0; k < CW; ++k) if (ch * CW + k > r) s[k] = -INFINITY;
      }
      // row maximum: 3-input max over this thread's half (4 independent chains), then
      // one shuffle with the thread holding the other half of the row
      static_assert(CW % 8 == 0, "half rows come in multiples of 8 columns");
      float mxa[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) mxa[q] = fmaxf(s[2 * q], s[2 * q + 1]);
#pragma unroll
      for (int k = 8; k < CW; k += 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) mxa[q] = max3(mxa[q], s[k + 2 * q], s[k + 2 * q + 1]);
      }
      const float mh = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
      const float mx = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));

      float alpha = 1.f;
      bool rescale = false;
      const float mxs = mx * p.scale_log2;
      m_true = fmaxf(m_true, mxs);
      if (j == 0) {
        m_ref = mxs;
      } else if (mxs > m_ref + kRescaleThreshold) {
        alpha = ex2(m_ref - mxs);
        l *= alpha;
        m_ref = mxs;
        rescale = true;
      }
      // P = exp2(s * scale_log2 - m_ref): packed fp32x2 FMA, MUFU ex2, packed sums
      const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
      uint64_t acc[4] = {0, 0, 0, 0};
      uint32_t pk[CW / 2];
#pragma unroll
      for (int k = 0; k < CW; k += 2) {
        const uint64_t x = f2_fma(f2_pack(s[k], s[k + 1]), scale2, negm2);
        float x0, x1;
        f2_unpack(x, x0, x1);
        const float e0 = ex2(x0), e1 = ex2(x1);
        acc[(k >> 1) & 3] = f2_add(acc[(k >> 1) & 3], f2_pack(e0, e1));
        pk[k >> 1] = row_ok ? pack_bf16(e0, e1) : 0u;
      }
      {
        const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        float t0, t1;
        f2_unpack(t, t0, t1);
        l += t0 + t1;
      }
      // P (bf16 pairs) over the first BLOCK/2 columns of the S buffer; the S columns it
      // overwrites were read by this same warp above
      if constexpr (CW == 64) tmem_st32s<CW / 2>(sbase, pk);
      else tmem_st16s<CW / 2>(sbase, pk);
      if (__any_sync(0xffffffffu, rescale)) {
        // O may be touched only once PV of the previous block is complete
        const uint32_t gp = G - 1, pb = gp % kSBufs;
        if (!warp_wait_bar(c, smem_u32(&c->pv_done[pb]), (gp / kSBufs) & 1, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < DW / 32; ++cc) {
          uint32_t t[32];
          tmem_ld32s_wait<DW>(lane_base + cc * 32, t);
#pragma unroll
          for (int q = 0; q < 32; ++q) t[q] = __float_as_uint(__uint_as_float(t[q]) * alpha);
          tmem_st32s<DW>(lane_base + cc * 32, t);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&c->p_full[b]));
        if (pend_qs >= 0 && --pend_left == 0) release_pending();
      }
    }
    if (!ok) break;
    if (lane == 0 && pend_qs >= 0) release_pending();  // an item shorter than the deferral
    l += __shfl_xor_sync(0xffffffffu, l, 16);  // row sum over both halves
    // epilogue: wait for the last PV of this item; the next item's first PV waits for
    // these warps' P, which they store only after the reads below
    const uint32_t gl = G - 1;
    if (!warp_wait_bar(c, smem_u32(&c->pv_done[gl % kSBufs]), (gl / kSBufs) & 1, p.err)) break;
    tc_fence_after();
    uint32_t o[DW];
    if constexpr (DW == 64) tmem_ld64s_wait<DW>(lane_base, o);
    else tmem_ld32s_wait<DW>(lane_base, o);
    tc_fence_before();
    const uint32_t ii = items - 1;  // this item's place in the worklist; its Q buffer:
    const uint32_t qs = ii % kQBufs;
    const uint32_t qbuf = data + qs * C::kQBytes;
    // final mode: O / l in bf16 goes into the item's Q buffer (its S products are
    // complete) in the 128-byte-swizzled layout of the output tensor map, and leaves by
    // one TMA store; partial outputs are written directly
    const bool tma_out = !partial && !(UNITS && pslot >= 0);
    if (row_ok) {
      const float* of = reinterpret_cast<const float*>(o);
      constexpr float kLn2 = 0.693147180559945309f;
      if (!tma_out) {  // unnormalised partial of a KV shard or of a piece
        const bool piece = UNITS && pslot >= 0;
        const long long prow = piece ? (long long)pslot * BLOCK + r : grow;
        const float f = ex2(m_ref - m_true);
        float4* dst = reinterpret_cast<float4*>((piece ? p.o_piece : p.o_part) + prow * D + ch * DW);
#pragma unroll
        for (int i = 0; i < DW / 4; ++i)
          dst[i] = make_float4(of[4 * i] * f, of[4 * i + 1] * f, of[4 * i + 2] * f, of[4 * i + 3] * f);
        if (ch == 0) {
          (piece ? p.m_piece : p.m_part)[prow] = m_true * kLn2;
          (piece ? p.l_piece : p.l_part)[prow] = l * f;
        }
      } else {
        const float inv = 1.f / l;
#pragma unroll
        for (int i = 0; i < DW / 8; ++i) {
          const int col = ch * DW + 8 * i;  // 16 bytes of row r: unit (col % 64) / 8 of chunk col / 64
          const uint32_t addr =
              qbuf + (col >> 6) * C::kChunk128 + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4);
          st_shared_v4(addr, pack_bf16(of[8 * i + 0] * inv, of[8 * i + 1] * inv),
                       pack_bf16(of[8 * i + 2] * inv, of[8 * i + 3] * inv),
                       pack_bf16(of[8 * i + 4] * inv, of[8 * i + 5] * inv),
                       pack_bf16(of[8 * i + 6] * inv, of[8 * i + 7] * inv));
        }
        if (ch == 0 && p.lse) p.lse[grow] = (m_ref + __log2f(l)) * kLn2;
      }
    }
    // one thread per item (the softmax warps take turns) releases the Q buffer: in final
    // mode once the output tile has been stored from it
    // (every item completes one phase of epi_full of its buffer, whatever the mode)
    const bool releaser = warp == kSoftmaxWarp0 + (int)(ii % 8) && lane == 0;
    if (tma_out) fence_proxy_async_smem();  // the generic-proxy writes above, before the TMA store
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&c->epi_full[qs]));
    if (releaser) {
      if (wait_bar(c, smem_u32(&c->epi_full[qs]), (ii / kQBufs) & 1, p.err) && tma_out) {
        const int row0 = (int)(bh * p.S + (long long)qb * BLOCK);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) tma_store_2d(to, qbuf + cc * C::kChunk128, cc * 64, row0);
        bulk_commit_group();
        pend_qs = (int)qs;
        pend_left = kDeferRelease;
        if (kDeferRelease == 0) release_pending();
      } else {
        mbar_arrive(smem_u32(&c->q_empty[qs]));
      }
    }
  }
  if (lane == 0 && pend_qs >= 0) release_pending();
  if (lane == 0) bulk_wait_all();  // the output stores this warp issued are complete
}

template <int BLOCK, int D, bool UNITS>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to, const AttnParams p) {
  using C = Cfg<BLOCK, D>;
  extern __shared__ uint8_t smem_raw[];
  // shared memory: Q buffers | K ring | V ring | control
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* c = reinterpret_cast<Ctrl*>(base + C::kDataBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t_start = globaltimer();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(smem_u32(&c->q_full[i]), 1);
      // the S issuer's commit (its MMAs read the Q tile) and the item's epilogue (in final
      // mode the output tile passes through this buffer on its way out)
      mbar_init(smem_u32(&c->q_empty[i]), 2);
      mbar_init(smem_u32(&c->epi_full[i]), 8);  // 8 softmax warps
    }
    for (int i = 0; i < kKStages; ++i) mbar_init(smem_u32(&c->k_full[i]), 1);
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_u32(&c->s_full[i]), 1);
      mbar_init(smem_u32(&c->p_full[i]), 9);  // 8 softmax warps + the V producer
      mbar_init(smem_u32(&c->pv_done[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&c->item_full[i]), 1);
      mbar_init(smem_u32(&c->item_empty[i]), 10);  // both MMA issuers + 8 softmax warps
    }
    mbar_init(smem_u32(&c->drain), 2);  // one commit per MMA issuer
    c->abort_flag = 0;
    c->blocks_done = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&to);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&c->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  griddep_wait();  // worklist, mask and Q/K/V may come from the previous grid

  if (warp < kSoftmaxWarp0) {
    setmaxnreg_dec<kRegsControl>();
    if (warp < 2) {
      if (!UNITS && p.dense_cols)
        run_producer_listed<BLOCK, D>(warp, &tq, &tk, &tv, p, c, base);
      else
        run_producer<BLOCK, D, UNITS>(warp, &tq, &tk, &tv, p, c, base);
    } else {
      if (lane == 0) {
        if (warp == kMmaWarp) run_mma_s<BLOCK, D>(p, c, smem_u32(base), tmem);
        else run_mma_pv<BLOCK, D>(p, c, smem_u32(base), tmem);
        drain_bar(smem_u32(&c->drain), 0);  // both issuers' MMAs are complete
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    run_softmax<BLOCK, D, UNITS>(p, c, tmem, smem_u32(base), &to);
  }
  griddep_launch_dependents();  // this CTA's work is done; the next grid may start its prologue

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && p.timing) {
    p.timing[3 * blockIdx.x + 0] = (int64_t)t_start;
    p.timing[3 * blockIdx.x + 1] = (int64_t)globaltimer();
    p.timing[3 * blockIdx.x + 2] = c->blocks_done;
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int encode_map(CUtensorMap* map, const void* ptr, long long rows, int d, int block) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return DBSP_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)block};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DBSP_OK : DBSP_ERR_CUDA;
}

template <int BLOCK, int D, bool UNITS>
int launch_attn_t(const void* q, const void* k, const void* v, const AttnParams& p, long long rows,
                  int n_workers, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  if (encode_map(&tq, q, rows, D, BLOCK) || encode_map(&tk, k, rows, D, BLOCK) ||
      encode_map(&tv, v, rows, D, BLOCK))
    return dbsp::cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  // final mode: the bf16 output tile leaves shared memory by a TMA store (partial mode: unused)
  if (encode_map(&to, p.out ? static_cast<const void*>(p.out) : q, rows, D, BLOCK))
    return dbsp::cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(out)");
  constexpr size_t smem = smem_bytes<BLOCK, D>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  auto kernel = attn_fwd_kernel<BLOCK, D, UNITS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaFuncSetAttribute(attn)");
  e = dbsp::launch_overlapped(kernel, dim3(n_workers), dim3(kThreads), smem, stream, tq, tk, tv, to, p);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "launch attn_fwd");
  return DBSP_OK;
}

// The unit logic is compiled only into the kernels that take a unit table, so the
// plain worklist path carries none of it.
template <int BLOCK, int D>
int launch_attn(const void* q, const void* k, const void* v, const AttnParams& p, long long rows,
                int n_workers, cudaStream_t stream) {
  return p.unit_item ? launch_attn_t<BLOCK, D, true>(q, k, v, p, rows, n_workers, stream)
                     : launch_attn_t<BLOCK, D, false>(q, k, v, p, rows, n_workers, stream);
}

}  // namespace

namespace {

struct Units {
  const int32_t* item;
  const int32_t* pk;
  const int32_t* slot;
  int n;
  int max_slots;
  float* o_piece;
  float* m_piece;
  float* l_piece;
  const int32_t* dense_n = nullptr;     // dense-block lists (plain worklists only)
  const uint16_t* dense_cols = nullptr;
};

int attn_fwd(const void* q, const void* k, const void* v, const uint8_t* mask, int B, int H, int S, int d,
             int block, int causal, float scale, const int32_t* worker_offsets, const int32_t* worklist,
             int n_workers, void* out, float* lse, float* o_part, float* m_part, float* l_part,
             int64_t* cta_timing, const Units& u, void* stream) {
  if (!q || !k || !v || !mask || !worker_offsets || !worklist) return DBSP_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || n_workers < 1 || n_workers > (1 << 20)) return DBSP_ERR_INVALID_ARG;
  const bool final_mode = out != nullptr;
  const bool partial_mode = o_part != nullptr || m_part != nullptr || l_part != nullptr;
  if (final_mode == partial_mode) return DBSP_ERR_INVALID_ARG;
  if (partial_mode && (!o_part || !m_part || !l_part)) return DBSP_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || (block != 64 && block != 128)) return DBSP_ERR_UNSUPPORTED;
  if (S % block != 0) return DBSP_ERR_UNSUPPORTED;
  const long long rows = (long long)B * H * S;
  const long long n_items = (long long)B * H * (S / block);
  if (rows >= (1LL << 31) || n_items * (S / block) >= (1LL << 40)) return DBSP_ERR_INVALID_ARG;
  if (!dbsp::aligned(q, 16) || !dbsp::aligned(k, 16) || !dbsp::aligned(v, 16) ||
      (out && !dbsp::aligned(out, 16)) || (o_part && !dbsp::aligned(o_part, 16)) ||
      (lse && !dbsp::aligned(lse, 4)) || (m_part && !dbsp::aligned(m_part, 4)) ||
      (l_part && !dbsp::aligned(l_part, 4)) || (cta_timing && !dbsp::aligned(cta_timing, 8)) ||
      (u.o_piece && !dbsp::aligned(u.o_piece, 16)) || (u.m_piece && !dbsp::aligned(u.m_piece, 4)) ||
      (u.l_piece && !dbsp::aligned(u.l_piece, 4)))
    return DBSP_ERR_INVALID_ARG;
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt((float)d);

  AttnParams p;
  p.mask = mask;
  p.H = H;
  p.S = S;
  p.nQ = S / block;
  p.nK = S / block;
  p.n_items = (int)n_items;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.offsets = worker_offsets;
  p.worklist = worklist;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = final_mode ? lse : nullptr;
  p.o_part = o_part;
  p.m_part = m_part;
  p.l_part = l_part;
  p.timing = cta_timing;
  p.err = dbsp::error_word(dev);
  p.unit_item = u.item;
  p.unit_pk = u.pk;
  p.unit_slot = u.slot;
  p.n_units = u.n;
  p.max_slots = u.max_slots;
  p.o_piece = u.o_piece;
  p.m_piece = u.m_piece;
  p.l_piece = u.l_piece;
  p.dense_n = u.dense_n;
  p.dense_cols = u.dense_cols;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (block == 128 && d == 128) return launch_attn<128, 128>(q, k, v, p, rows, n_workers, s);
  if (block == 128 && d == 64) return launch_attn<128, 64>(q, k, v, p, rows, n_workers, s);
  if (block == 64 && d == 128) return launch_attn<64, 128>(q, k, v, p, rows, n_workers, s);
  return launch_attn<64, 64>(q, k, v, p, rows, n_workers, s);
}

}  // namespace

extern "C" int dbsp_block_sparse_attn_fwd(const void* q, const void* k, const void* v,
                                          const uint8_t* mask, int B, int H, int S, int d,
                                          int block, int causal, float scale,
                                          const int32_t* worker_offsets, const int32_t* worklist,
                                          int n_workers, void* out, float* lse, float* o_part,
                                          float* m_part, float* l_part, int64_t* cta_timing,
                                          void* stream) {
  const Units none{nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, nullptr};
  return attn_fwd(q, k, v, mask, B, H, S, d, block, causal, scale, worker_offsets, worklist, n_workers, out,
                  lse, o_part, m_part, l_part, cta_timing, none, stream);
}

extern "C" int dbsp_block_sparse_attn_fwd_units(const void* q, const void* k, const void* v,
                                                const uint8_t* mask, int B, int H, int S, int d,
                                                int block, int causal, float scale,
                                                const int32_t* worker_offsets, const int32_t* worklist,
                                                int n_workers, const int32_t* unit_item,
                                                const int32_t* unit_pk, const int32_t* unit_slot,
                                                int n_units, void* out, float* lse, float* o_piece,
                                                float* m_piece, float* l_piece, int max_slots,
                                                int64_t* cta_timing, void* stream) {
  if (!unit_item || !unit_pk || !unit_slot || n_units < 0 || max_slots < 0 || !out) return DBSP_ERR_INVALID_ARG;
  if (!o_piece || !m_piece || !l_piece) return DBSP_ERR_INVALID_ARG;
  const Units u{unit_item, unit_pk, unit_slot, n_units, max_slots, o_piece, m_piece, l_piece};
  return attn_fwd(q, k, v, mask, B, H, S, d, block, causal, scale, worker_offsets, worklist, n_workers, out,
                  lse, nullptr, nullptr, nullptr, cta_timing, u, stream);
}

extern "C" int dbsp_block_sparse_attn_fwd_listed(const void* q, const void* k, const void* v,
                                                 const uint8_t* mask, int B, int H, int S, int d,
                                                 int block, int causal, float scale,
                                                 const int32_t* worker_offsets, const int32_t* worklist,
                                                 int n_workers, const int32_t* dense_n,
                                                 const uint16_t* dense_cols, void* out, float* lse,
                                                 float* o_part, float* m_part, float* l_part,
                                                 int64_t* cta_timing, void* stream) {
  if (!dense_n || !dense_cols || !dbsp::aligned(dense_n, 4) || !dbsp::aligned(dense_cols, 2))
    return DBSP_ERR_INVALID_ARG;
  Units u{nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, nullptr};
  u.dense_n = dense_n;
  u.dense_cols = dense_cols;
  return attn_fwd(q, k, v, mask, B, H, S, d, block, causal, scale, worker_offsets, worklist, n_workers, out,
                  lse, o_part, m_part, l_part, cta_timing, u, stream);
}
