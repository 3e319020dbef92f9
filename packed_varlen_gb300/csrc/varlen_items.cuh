// Work items of the packed varlen attention kernels (head dim 64 on single
// CTAs, head dim 128 on CTA pairs): their parameters, the decode of item i of
// the length-ordered list into rows and keys, and the key-tile order.  Both
// kernels take a work item of kVarlenItemRows query rows of one (sequence,
// head) and walk its keys in kVarlenTile-key tiles in the same order, so a
// sequence's rows come out the same whatever the batch around it.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sched.cuh"

namespace pa {

constexpr int kVarlenTile = 128;       // keys of a K/V tile, rows of a Q tile
constexpr int kVarlenItemRows = 256;   // query rows of a work item

struct VarlenParams {
  __nv_bfloat16 *out;
  const int32_t *cu_q, *cu_k;
  int batch, H, total_q, total_k, max_q, max_k;
  float scale_log2;
  int32_t *status;
};

struct ItemInfo {
  int q_row0;   // global row of the item's first query
  int rows;     // valid query rows in the item (1..kVarlenItemRows)
  int k0;       // global row of the sequence's first key
  int lk;       // keys of the sequence
  int nk;       // key tiles
  int head;
  int rot;      // first key tile visited
};

// Key tile visited j-th.  Items start at key tile (item index in the
// sequence mod nk) and wrap around, so the workers of a wave, which hold
// consecutive query blocks of one head, read different K/V tiles at any
// moment.  The order depends only on the sequence's own lengths and the
// item's position in it, so a sequence's result is the same in any batch.
__device__ __forceinline__ int key_tile(const ItemInfo &it, int j) {
  const int kt = it.rot + j;
  return kt >= it.nk ? kt - it.nk : kt;
}

// Item i (0 <= i < prefix[batch]) of the work list; a sequence whose
// boundaries are invalid reads as empty (the list build records why).
__device__ __forceinline__ ItemInfo item_info(const VarlenParams &p, const int32_t *order,
                                              const int32_t *prefix, int i) {
  const WorkItem w = sched_item(order, prefix, p.batch, p.H, i);
  int err;
  const SeqBounds sb = seq_bounds(p.cu_q, p.cu_k, w.seq, p.total_q, p.total_k, p.max_q,
                                  p.max_k, err);
  ItemInfo it;
  it.q_row0 = sb.q0 + w.tile * kVarlenItemRows;
  it.rows = min(kVarlenItemRows, sb.lq - w.tile * kVarlenItemRows);
  it.k0 = sb.k0;
  it.lk = sb.lk;
  it.nk = (sb.lk + kVarlenTile - 1) / kVarlenTile;
  it.head = w.head;
  it.rot = it.nk > 0 ? w.tile % it.nk : 0;
  return it;
}

}  // namespace pa
