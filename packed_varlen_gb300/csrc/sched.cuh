// Length-ordered work list over (sequence, head, q_tile) items, rebuilt by
// every CTA from cu_seqlens in shared memory.  No workspace, no atomics, no
// host round trip: a CTA of a persistent kernel takes items
// blockIdx.x, blockIdx.x + gridDim.x, ... of this list.
//
// Order: sequences by key length, longest first (ties: lower index first),
// then heads in order, then query tiles in order.  The longest request
// dominates a mixed batch and the per-bucket loop it replaces left bubbles
// ("[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
// varlen attention for mixfusion", Purpose), so the heaviest items start
// first; consecutive items share a head, so the CTAs of one wave stream the
// same K/V rows through L2.
#pragma once

#include <stdint.h>

#include "packedattn.h"

namespace pa {

__device__ __forceinline__ void record_error(int32_t *status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Validated boundaries of one sequence.
struct SeqBounds {
  int32_t q0, lq, k0, lk;
};

// Reads and checks sequence b's boundaries.  A sequence whose boundaries
// break 0 <= cu[b] <= cu[b+1] <= total (with cu[0] == 0) or whose length
// exceeds max_q / max_k is returned empty; `err` receives the reason.
__device__ __forceinline__ SeqBounds seq_bounds(const int32_t *__restrict__ cu_q,
                                                const int32_t *__restrict__ cu_k, int b,
                                                int total_q, int total_k, int max_q,
                                                int max_k, int &err) {
  const int q0 = __ldg(cu_q + b), q1 = __ldg(cu_q + b + 1);
  const int k0 = __ldg(cu_k + b), k1 = __ldg(cu_k + b + 1);
  const bool okq = (q0 >= 0) && (q0 <= q1) && (q1 <= total_q) && (b > 0 || q0 == 0);
  const bool okk = (k0 >= 0) && (k0 <= k1) && (k1 <= total_k) && (b > 0 || k0 == 0);
  SeqBounds s{0, 0, 0, 0};
  err = 0;
  if (!(okq && okk)) {
    err = PA_DEVICE_ERR_CU_SEQLENS;
  } else if (q1 - q0 > max_q || k1 - k0 > max_k) {
    err = PA_DEVICE_ERR_MAX_LEN;
  } else {
    s.q0 = q0;
    s.lq = q1 - q0;
    s.k0 = k0;
    s.lk = k1 - k0;
  }
  return s;
}

// Builds the list in shared memory.  order[batch], prefix[batch + 1] persist;
// tmp_lq / tmp_lk [batch] are only used during the build (they may alias
// memory the caller reuses afterwards).  All threads of the CTA call it; it
// ends with __syncthreads().  Item count = prefix[batch].
__device__ inline void sched_build(int32_t *order, int32_t *prefix, int32_t *tmp_lq,
                                   int32_t *tmp_lk, const int32_t *__restrict__ cu_q,
                                   const int32_t *__restrict__ cu_k, int batch, int H,
                                   int tile_m, int total_q, int total_k, int max_q,
                                   int max_k, int32_t *status, bool report) {
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int b = tid; b < batch; b += nt) {
    int err;
    const SeqBounds sb = seq_bounds(cu_q, cu_k, b, total_q, total_k, max_q, max_k, err);
    if (err && report) record_error(status, err);
    tmp_lq[b] = sb.lq;
    tmp_lk[b] = sb.lk;
  }
  __syncthreads();
  // Rank sort by (key length descending, index ascending).
  for (int b = tid; b < batch; b += nt) {
    const int lb = tmp_lk[b];
    int rank = 0;
    for (int j = 0; j < batch; ++j) {
      const int lj = tmp_lk[j];
      rank += (lj > lb) || (lj == lb && j < b);
    }
    order[rank] = b;
  }
  __syncthreads();
  // Exclusive prefix of item counts in taken order (warp 0, 32 at a time).
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base < batch; base += 32) {
      const int idx = base + tid;
      int cnt = 0;
      if (idx < batch) cnt = H * ((tmp_lq[order[idx]] + tile_m - 1) / tile_m);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += y;
      }
      if (idx < batch) prefix[idx] = carry + incl - cnt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) prefix[batch] = carry;
  }
  __syncthreads();
}

struct WorkItem {
  int32_t seq, head, tile;
};

// Item i (0 <= i < prefix[batch]) -> (sequence, head, q_tile).
__device__ __forceinline__ WorkItem sched_item(const int32_t *order, const int32_t *prefix,
                                               int batch, int H, int i) {
  int lo = 0, hi = batch;  // largest s < batch with prefix[s] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= i) lo = mid; else hi = mid;
  }
  const int ntiles = (prefix[lo + 1] - prefix[lo]) / H;
  const int r = i - prefix[lo];
  WorkItem w;
  w.seq = order[lo];
  w.head = r / ntiles;
  w.tile = r - w.head * ntiles;
  return w;
}

}  // namespace pa
