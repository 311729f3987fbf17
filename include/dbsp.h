/*
 * dbsp.h -- C ABI of libdbsp.so: load-balanced block-sparse attention forward on
 * one GB300 (sm_103a).
 *
 * The operations follow two web pages:
 *   [db-SP blog]  "db-SP：稀疏注意力头并行和序列并行的负载均衡问题"
 *                 (yjmstr.github.io, 2026-01-30), scenarios 1 and 2;
 *   [6D notes]    "6D 并行下的 Attention Kernel 与通信重叠" (walkerchi.com),
 *                 §2.1 ring-attention pseudocode and §2.3 causal / striped.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are caller-owned DEVICE memory unless stated otherwise (e.g. a torch
 *   tensor's data_ptr()). The library never frees or keeps them, and allocates no
 *   device memory per call. It keeps one device error word per device (a static
 *   __device__ variable) and caches nothing else that refers to caller memory.
 * - `stream` is a cudaStream_t (NULL = legacy default stream). Every call only
 *   enqueues work on it and returns; results are ready when the stream is.
 * - Arguments are validated on the host before anything touches the GPU:
 *   DBSP_ERR_INVALID_ARG for a bad size, NULL or misaligned pointer,
 *   DBSP_ERR_UNSUPPORTED for a shape the kernels do not implement or a device
 *   that is not sm_103, DBSP_ERR_CUDA for a failed launch (the CUDA error is
 *   cleared and its text is kept for dbsp_last_error_string()).
 * - Problems the kernels can only see in device data (a negative load, an item
 *   id out of range in a worklist, a pipeline wait that timed out) set the
 *   device error word instead of faulting; dbsp_device_status() reports it.
 * - Integer outputs are exact; there is exactly one correct worklist.
 * - No CPU fallback exists: every call either launches its kernel or fails.
 */
#ifndef DBSP_H
#define DBSP_H

#include <stdint.h>

#if defined(__GNUC__)
#define DBSP_API __attribute__((visibility("default")))
#else
#define DBSP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DBSP_OK = 0,
  DBSP_ERR_INVALID_ARG = 1,
  DBSP_ERR_UNSUPPORTED = 2,
  DBSP_ERR_CUDA = 3,
  DBSP_ERR_TIMEOUT = 4
} dbsp_status;

/* Largest worker count dbsp_plan_lpt accepts (one warp holds 32 loads per lane). */
#define DBSP_MAX_WORKERS 1024

/* Static text for a status code. Never NULL. */
DBSP_API const char* dbsp_status_string(int status);

/* Text of the last DBSP_ERR_CUDA raised on the calling thread ("" if none). */
DBSP_API const char* dbsp_last_error_string(void);

/*
 * Mask loads.  [db-SP blog, scenario 2, first bullet]: the load of a Q-block is
 * the number of dense (non-zero) blocks in its row of the head's block mask, the
 * load of a KV-block the number in its column. [db-SP blog, scenario 1]: a head's
 * load is its total number of dense blocks.
 *
 *   mask        uint8 [B, H, nQ, nK], row-major; any non-zero byte is dense.
 *   row_loads   int32 [B, H, nQ]  out: dense blocks per Q-block row.
 *   col_loads   int32 [B, H, nK]  out: dense blocks per KV-block column.
 *   head_loads  int32 [B, H]      out, may be NULL.
 * Requires B, H, nQ, nK >= 1 and B*H*nQ*nK < 2^31; nQ > 131072 or nK > 16384
 * returns DBSP_ERR_UNSUPPORTED. Output buffers must not overlap the mask. Exact
 * integer results; one kernel launch. A copy of mask rows that does not arrive
 * within 2 s sets DBSP_ERR_TIMEOUT on the device.
 */
DBSP_API int dbsp_block_mask_loads(const uint8_t* mask, int B, int H, int nQ, int nK,
                          int32_t* row_loads, int32_t* col_loads, int32_t* head_loads,
                          void* stream);

/*
 * Mask loads of causal attention.  [6D attention notes §2.3]: under a causal mask the
 * KV blocks after a Q block's diagonal are skipped, so only the dense blocks on or below
 * the diagonal (column <= row) are work. As dbsp_block_mask_loads, counting only those:
 * the loads of a mask that was not clipped to the diagonal beforehand, which is what
 * dbsp_plan_lpt should balance for dbsp_block_sparse_attn_fwd with causal = 1.
 * Requires nQ == nK (otherwise DBSP_ERR_INVALID_ARG); every other argument and limit as
 * in dbsp_block_mask_loads.
 */
DBSP_API int dbsp_block_mask_loads_causal(const uint8_t* mask, int B, int H, int nQ, int nK,
                                          int32_t* row_loads, int32_t* col_loads, int32_t* head_loads,
                                          void* stream);

/*
 * KV-block loads across heads.  [db-SP blog, scenario 2]: a KV-block's load is the
 * number of dense blocks in its mask column; when the KV sequence is split into
 * shards shared by every head (sequence parallelism), the load that a shard
 * receives from block j is the column count summed over all heads.
 *
 *   col_loads   int32 [groups, nK]  column loads, e.g. dbsp_block_mask_loads's
 *               col_loads with groups = B * H.
 *   kv_loads    int32 [nK]  out: kv_loads[j] = sum over g of col_loads[g, j].
 * Requires groups, nK >= 1 and groups * nK < 2^31. Exact; one kernel launch. The
 * result can be planned over shards with dbsp_plan_lpt (items = KV blocks,
 * workers = shards).
 */
DBSP_API int dbsp_kv_block_loads(const int32_t* col_loads, int groups, int nK, int32_t* kv_loads,
                                 void* stream);

/*
 * The block masks of KV shards.  [db-SP blog, scenario 2]: when the KV sequence is
 * split into shards, each shard's pass attends only to the KV blocks it holds. Given
 * the shard of every KV block (e.g. worker_of of dbsp_plan_lpt over dbsp_kv_block_loads),
 * out[s] is mask with every column j of another shard (shard_of[j] != s) cleared.
 *
 *   mask      uint8 [B, H, nQ, nK]
 *   shard_of  int32 [nK], values in [0, n_shards); a value outside that range sets
 *             DBSP_ERR_INVALID_ARG on the device and clears column j in every shard.
 *   out       uint8 [n_shards, B, H, nQ, nK]  out; must not overlap mask.
 * Requires B, H, nQ, nK, n_shards >= 1, n_shards <= 65535 and B*H*nQ*nK < 2^31. The
 * mask is read once; one kernel launch (16-byte accesses when nK % 16 == 0 and both
 * byte pointers are 16-byte aligned, byte by byte otherwise).
 */
DBSP_API int dbsp_shard_masks(const uint8_t* mask, int B, int H, int nQ, int nK, const int32_t* shard_of,
                              int n_shards, uint8_t* out, void* stream);

/*
 * Dense-block lists.  [db-SP blog, scenario 2, first bullet]: a Q-block row's load is
 * its dense blocks; this lists them. For every row r = (b*H + h)*nQ + qb of the mask,
 * the KV-block indices of its dense blocks in ascending order go to
 * cols[r*nK + 0 .. counts[r] - 1] (with causal != 0 only the blocks on or below the
 * diagonal, the ones causal attention computes). Input for the attention producers
 * (dbsp_block_sparse_attn_fwd_listed), which then read an item's tiles from here
 * instead of scanning its mask row.
 *
 *   mask    uint8 [B, H, nQ, nK]; any non-zero byte is a dense block.
 *   counts  int32 [B*H*nQ] out: the row's dense blocks (= its row load).
 *   cols    uint16 [B*H*nQ, nK] out, 2-byte aligned; entries past counts[r] are not
 *           written.
 * Requires B, H, nQ, nK >= 1, B*H*nQ*nK < 2^31, nK <= 65536 (else DBSP_ERR_UNSUPPORTED)
 * and nQ == nK with causal != 0. One warp per row, 16-byte loads when nK % 16 == 0 and
 * the mask is 16-byte aligned, byte loads otherwise. Ownership: caller-owned buffers.
 */
DBSP_API int dbsp_dense_block_lists(const uint8_t* mask, int B, int H, int nQ, int nK, int causal,
                                    int32_t* counts, uint16_t* cols, void* stream);

/*
 * LPT plan with stay-in-place bonus.  [db-SP blog, scenario 1]: repeatedly give
 * the largest remaining item to the currently least-loaded worker (LPT).
 * [db-SP blog, scenario 2, third bullet]: an item placed on its original worker
 * counts as lighter when choosing.
 *
 * Items are taken in order of load descending, equal loads by id ascending. Item
 * i goes to the worker p minimising (L_p - stay_bonus * [p == home[i]], p); then
 * L_p += loads[i] (the true load). Ties go to the lowest worker index.
 *
 *   loads          int32 [n_items], each >= 0.
 *   home           int32 [n_items] with values in [0, n_workers), or NULL (no bonus).
 *   n_items        >= 0;  n_workers in [1, DBSP_MAX_WORKERS];  stay_bonus >= 0.
 *   worker_of      int32 [n_items]      out: worker of each item.
 *   worker_offsets int32 [n_workers+1]  out: CSR offsets into worklist.
 *   worklist       int32 [n_items]      out: item ids grouped by worker, each
 *                                       group in assignment order.
 *   worker_loads   int64 [n_workers]    out, may be NULL: accrued true loads.
 * Limits: n_items * n_workers < 2^31; either max(loads) <= 32767 or
 * n_items <= 16384 (otherwise the device error word is set to
 * DBSP_ERR_UNSUPPORTED). A negative load or out-of-range home sets
 * DBSP_ERR_INVALID_ARG on the device. One single-CTA kernel launch; the output
 * arrays double as the kernel's working storage.
 */
DBSP_API int dbsp_plan_lpt(const int32_t* loads, const int32_t* home, int n_items, int n_workers,
                  int32_t stay_bonus, int32_t* worker_of, int32_t* worker_offsets,
                  int32_t* worklist, int64_t* worker_loads, void* stream);

/*
 * LPT plan over planning loads loads[i] * block_cost + item_cost.  The pages count
 * work in dense blocks ([db-SP blog, scenario 2, first bullet]), which is
 * dbsp_plan_lpt (block_cost = 1, item_cost = 0). On one GPU an item also costs
 * something of its own (its Q tile, its epilogue): with item_cost > 0 items without
 * dense blocks no longer all land on the least-loaded worker. The transform keeps
 * the order of the items (block_cost >= 1), so only the worker choice changes.
 *
 *   block_cost in [1, 65535], item_cost in [0, 2^24]; every other argument as in
 *   dbsp_plan_lpt, and worker_loads accrues the planning loads. A planning load of
 *   2^31 or more sets DBSP_ERR_UNSUPPORTED on the device.
 */
DBSP_API int dbsp_plan_lpt_cost(const int32_t* loads, const int32_t* home, int n_items, int n_workers,
                       int32_t stay_bonus, int32_t block_cost, int32_t item_cost,
                       int32_t* worker_of, int32_t* worker_offsets, int32_t* worklist,
                       int64_t* worker_loads, void* stream);

/*
 * LPT plan (as dbsp_plan_lpt_cost, no bonus) over the first *n_items_dev items, the
 * count living in device memory (e.g. counts[0] of dbsp_split_plan), so that a
 * plan over a unit table needs no host synchronisation.
 *
 *   n_items_dev   int32 [1] device pointer: the item count, clamped to [0, n_items_max].
 *   n_items_max   >= 0: the capacity of loads, worker_of and worklist.
 * Every other argument as in dbsp_plan_lpt_cost; worklist and worker_offsets cover
 * the first *n_items_dev items only.
 */
DBSP_API int dbsp_plan_lpt_cost_n(const int32_t* loads, const int32_t* n_items_dev, int n_items_max,
                         int n_workers, int32_t block_cost, int32_t item_cost, int32_t* worker_of,
                         int32_t* worker_offsets, int32_t* worklist, int64_t* worker_loads,
                         void* stream);

/*
 * Split plan: heavy items cut into pieces along their KV blocks.  [db-SP blog,
 * scenario 1]: the greedy cannot balance perfectly, partly because an item's load
 * cannot be divided; the page's closing remark points at splitting the load
 * further. Item i with load L = loads[i] > T becomes k = min(ceil(L / T), max_pieces)
 * pieces; piece j takes the row's dense blocks whose rank (column order, within the
 * causal limit) lies in [floor(j L / k), floor((j + 1) L / k)). Every other item
 * stays whole (k = 1).
 *
 *   loads          int32 [n_items] >= 0 (dense blocks per item within its causal
 *                  limit, e.g. row loads of dbsp_block_mask_loads for a causal mask
 *                  without blocks above the diagonal).
 *   n_workers      >= 1: used by the automatic T.
 *   max_piece_load T; <= 0 selects T = ceil(ceil(total / n_workers) / 2).
 *   max_pieces     in [1, 1024];  max_slots >= 0: capacity for pieces.
 * Outputs (device, written by one single-CTA kernel):
 *   unit_item, unit_pk, unit_slot, unit_load  int32 [n_items * max_pieces]: the
 *                  unit table. Units [0, n_whole) are the whole items in item order
 *                  (pk = 1 << 16, slot = -1); unit n_whole + s is piece slot s, the
 *                  pieces of each split item consecutive in j (pk = j | k << 16).
 *                  unit_load: the unit's dense blocks.
 *   split_item     int32 [n_items]: the split items in item order.
 *   split_off      int32 [n_items + 1]: slots of split item t are
 *                  split_off[t] .. split_off[t + 1] - 1.
 *   counts         int32 [5]: units U = n_whole + n_slots, n_whole, n_split,
 *                  n_slots, T.
 * A negative load sets DBSP_ERR_INVALID_ARG, more than max_slots pieces
 * DBSP_ERR_UNSUPPORTED, on the device; counts are then zero.
 */
DBSP_API int dbsp_split_plan(const int32_t* loads, int n_items, int n_workers, int32_t max_piece_load,
                    int32_t max_pieces, int32_t max_slots, int32_t* unit_item, int32_t* unit_pk,
                    int32_t* unit_slot, int32_t* unit_load, int32_t* split_item, int32_t* split_off,
                    int32_t* counts, void* stream);

/*
 * Block-sparse attention forward over an LPT worklist.  [6D notes §2.1, step 2]:
 * a chunk of keys yields the unnormalised output O, the row maximum m and the
 * row sum l of the softmax numerators; the result is O / l (last line of the
 * loop). Keys are admitted only in dense blocks of the mask ([db-SP blog,
 * scenario 2]); with causal != 0 a query sees keys at or before its position
 * ([6D notes §2.3]), blocks above the diagonal are skipped and the diagonal
 * block is masked element-wise.
 *
 *   q, k, v     bf16 [B, H, S, d] contiguous, 16-byte aligned.
 *   mask        uint8 [B, H, nQ, nK], nQ = nK = S / block.
 *   d in {64, 128}; block in {64, 128}; S % block == 0.
 *   scale       softmax scale; <= 0 selects 1/sqrt(d).
 *   worker_offsets, worklist, n_workers: a CSR worklist over items
 *               id = (b*H + h)*nQ + qb, e.g. from dbsp_plan_lpt. One CTA runs per
 *               worker, in list order. Items missing from the worklist are not
 *               written; an out-of-range id sets DBSP_ERR_INVALID_ARG on the device.
 * Final mode (out != NULL, o_part == NULL):
 *   out         bf16 [B, H, S, d]: O / l, rounded to nearest even.
 *   lse         fp32 [B, H, S] or NULL: m + ln(l) in natural-log units; rows with
 *               no admissible key get O = 0 and lse = -inf.
 * Partial mode (out == NULL; o_part, m_part, l_part all non-NULL; lse ignored):
 *   o_part      fp32 [B, H, S, d]: unnormalised O relative to the row maximum.
 *               Rows of items with no dense block are left unwritten: their
 *               (m, l) = (-inf, 0) marks them empty and no reader looks at them.
 *   m_part      fp32 [B, H, S]: row maximum of the scaled scores (-inf if empty).
 *   l_part      fp32 [B, H, S]: row sum of exp(score - m) (0 if empty).
 * cta_timing    int64 [n_workers * 3] or NULL: per worker the %globaltimer (ns)
 *               at start and end and the number of dense blocks processed.
 * Arithmetic: bf16 inputs, fp32 accumulation on the tensor cores; probabilities
 * are rounded to bf16 before the P.V product.
 */
DBSP_API int dbsp_block_sparse_attn_fwd(const void* q, const void* k, const void* v,
                               const uint8_t* mask, int B, int H, int S, int d, int block,
                               int causal, float scale,
                               const int32_t* worker_offsets, const int32_t* worklist,
                               int n_workers,
                               void* out, float* lse,
                               float* o_part, float* m_part, float* l_part,
                               int64_t* cta_timing, void* stream);

/*
 * dbsp_block_sparse_attn_fwd with the dense-block lists of dbsp_dense_block_lists: the
 * producer warps read each item's dense count and KV-block indices from dense_n and
 * dense_cols (same layout) instead of scanning its mask row, and fetch the next item's
 * entry while the current item's tiles go out; the mask is not read. Same arguments,
 * modes and results otherwise (bit-identical output). The lists must be those of the
 * same mask, built with the same causal flag. A count outside [0, limit] or an index at
 * or past the row's limit (nK, or qb + 1 when causal) sets DBSP_ERR_INVALID_ARG on the
 * device; the row is then written as empty, or the tile replaced by block 0.
 *   dense_n     int32 [B*H*nQ]; dense_cols uint16 [B*H*nQ, nK], 2-byte aligned.
 */
DBSP_API int dbsp_block_sparse_attn_fwd_listed(const void* q, const void* k, const void* v,
                                      const uint8_t* mask, int B, int H, int S, int d, int block,
                                      int causal, float scale,
                                      const int32_t* worker_offsets, const int32_t* worklist,
                                      int n_workers, const int32_t* dense_n,
                                      const uint16_t* dense_cols,
                                      void* out, float* lse,
                                      float* o_part, float* m_part, float* l_part,
                                      int64_t* cta_timing, void* stream);

/*
 * Block-sparse attention forward over a worklist of units (dbsp_split_plan).  Each
 * worklist entry u < n_units names piece j of k of item unit_item[u]
 * (unit_pk[u] = j | k << 16). A whole item (k = 1) is written to out / lse as in
 * dbsp_block_sparse_attn_fwd's final mode; a piece attends only to its dense blocks
 * (ranks [floor(j L / k), floor((j + 1) L / k)) of the row's L) and writes its
 * unnormalised partial, as in partial mode, to slot s = unit_slot[u]:
 *   o_piece  fp32 [max_slots, block, d]; m_piece, l_piece fp32 [max_slots, block]; a
 *            piece without dense blocks writes only (m, l) = (-inf, 0). A slot
 *            outside [0, max_slots) sets DBSP_ERR_INVALID_ARG and the unit is skipped.
 * The causal diagonal block, the last dense block of its row, is masked by the piece
 * that holds it (j = k - 1). Combine the pieces with dbsp_merge_pieces.
 * Every other argument as in dbsp_block_sparse_attn_fwd (final mode only). An entry
 * outside [0, n_units) or an inconsistent unit sets DBSP_ERR_INVALID_ARG on the
 * device.
 */
DBSP_API int dbsp_block_sparse_attn_fwd_units(const void* q, const void* k, const void* v,
                                     const uint8_t* mask, int B, int H, int S, int d, int block,
                                     int causal, float scale,
                                     const int32_t* worker_offsets, const int32_t* worklist,
                                     int n_workers, const int32_t* unit_item,
                                     const int32_t* unit_pk, const int32_t* unit_slot, int n_units,
                                     void* out, float* lse, float* o_piece, float* m_piece,
                                     float* l_piece, int max_slots, int64_t* cta_timing, void* stream);

/*
 * Merge of the pieces of split items.  [6D notes §2.1, step 3 and the final
 * division], as dbsp_merge_partials, over the slots of each split item: for split
 * item t (t < counts[2]) and row r of its Q-block, the partials at rows
 * s * block + r of o_piece / m_piece / l_piece, s in [split_off[t], split_off[t + 1]),
 * give out[item row r] (bf16) and lse (natural log; -inf and O = 0 when every piece
 * is empty). Rows of whole items are not touched.
 *
 *   split_item, split_off, counts: as written by dbsp_split_plan (device).
 *   max_slots  >= 0: capacity of the piece buffers, in slots (as given to
 *              dbsp_split_plan); no slot at or beyond it, nor beyond counts[3], is read.
 *   out bf16 [B, H, S, d], lse fp32 [B, H, S] or NULL; d in {64, 128}.
 * A split entry out of range (item, or slots outside [0, min(counts[3], max_slots)))
 * sets DBSP_ERR_INVALID_ARG on the device and its rows are skipped.
 */
DBSP_API int dbsp_merge_pieces(const float* o_piece, const float* m_piece, const float* l_piece,
                      const int32_t* split_item, const int32_t* split_off, const int32_t* counts,
                      int max_slots, int B, int H, int S, int d, int block, void* out, float* lse,
                      void* stream);

/* Size of the static piece scratch of dbsp_block_sparse_attn_fwd_split_noalloc. */
#define DBSP_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Split attention that allocates nothing.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory where they
 * run attention, such as a serving runtime whose memory pool is fixed up front, or a
 * host thread that may not call cudaMalloc (it synchronises the device). It runs
 * dbsp_block_sparse_attn_fwd_units and then dbsp_merge_pieces, with the pieces' fp32
 * O, m and l kept in a static device array of DBSP_NOALLOC_SCRATCH_BYTES (16 MiB)
 * that every GPU loading the library holds until the process exits, instead of
 * buffers passed by the caller. Inputs and outputs are still the caller's:
 *
 *   every argument as in dbsp_block_sparse_attn_fwd_units (final mode) and
 *   dbsp_merge_pieces; max_slots is the piece capacity given to dbsp_split_plan.
 * Limit: max_slots * block * (d + 2) * 4 bytes must not exceed
 * DBSP_NOALLOC_SCRATCH_BYTES (e.g. 252 slots at block = d = 128), else the call
 * returns DBSP_ERR_INVALID_ARG before touching the GPU.
 * The first call on a device, with that device current, looks up the array's device
 * address (cudaGetSymbolAddress) and caches it: make that first call before any
 * stream capture. No part of the scratch needs to start at zero: every piece writes
 * its m and l, and O is read only where l > 0. All calls share the one array and it
 * keeps the last call's contents, so calls that overlap on the GPU (e.g. on two
 * streams) race: order them on one stream or with events. Never calls cudaMalloc,
 * cudaFree or any allocating routine.
 */
DBSP_API int dbsp_block_sparse_attn_fwd_split_noalloc(
    const void* q, const void* k, const void* v, const uint8_t* mask, int B, int H, int S, int d, int block,
    int causal, float scale, const int32_t* worker_offsets, const int32_t* worklist, int n_workers,
    const int32_t* unit_item, const int32_t* unit_pk, const int32_t* unit_slot, int n_units,
    const int32_t* split_item, const int32_t* split_off, const int32_t* counts, int max_slots, void* out,
    float* lse, int64_t* cta_timing, void* stream);

/*
 * Merge of KV-shard partials.  [6D notes §2.1, step 3 and the final division]:
 * m* = max_k m_k, l = sum_k exp(m_k - m*) l_k, O = sum_k exp(m_k - m*) O_k / l.
 * A partial with l_k == 0 or m_k == -inf contributes nothing; a row whose
 * partials are all empty gets O = 0 and lse = -inf.
 *
 *   o_parts  fp32 [n_shards, rows, d];  m_parts, l_parts fp32 [n_shards, rows].
 *   out      bf16 [rows, d];  lse fp32 [rows] or NULL.
 * n_shards >= 1, rows >= 0, d a multiple of 4 in [4, 1024], 16-byte aligned
 * o_parts and 8-byte aligned out.
 */
DBSP_API int dbsp_merge_partials(const float* o_parts, const float* m_parts, const float* l_parts,
                        int n_shards, int64_t rows, int d, void* out, float* lse,
                        void* stream);

/*
 * Synchronises `stream`, then returns and clears the current device's error word
 * (DBSP_OK if no kernel reported a problem since the last call).
 */
DBSP_API int dbsp_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DBSP_H */
