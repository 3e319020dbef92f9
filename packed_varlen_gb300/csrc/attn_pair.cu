// Packed variable-length attention, head dim 128, on cta_group::2 CTA pairs.
//
// Computes, per sequence b, head h and query row i of b, softmax attention
// over the key rows of the same sequence only (the flat varlen path of
// "[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
// varlen attention for mixfusion", Key changes; "feat: Support dynamic
// batching for heterogeneous diffusion requests", AttentionMetadata).
//
// Design: persistent CTAs in clusters of two.  A work item is 256 query rows
// of one (sequence, head); the even CTA of the pair holds rows 0-127 and the
// odd CTA rows 128-255, and every MMA spans the pair (M = 256):
//   S = Q K^T   each CTA holds its Q tile and one 64-key half of the K tile
//               (keys 0-63 in the even CTA, 64-127 in the odd one);
//   O += P V    P comes from each CTA's own TMEM, and each CTA holds one
//               64-column half of the V tile (all 128 keys).
// Each CTA thus stages half of every K/V tile, and its TMEM carries a single
// 128-row O accumulator, which leaves room for three S buffers: the S of key
// tile g + 3 is issued right after the PV of tile g, so the softmax of the
// next tile never waits for the PV of the current one, and at an item's end
// the next item's first scores are already computed.
//   warp 0      TMA producer (both CTAs): Q once per item into one of two Q
//               buffers, then K0 K1 K2 V0 K3 V1 K4 V2 ... (the MMA issue
//               order) through a ring of 16 KB slots.  Both CTAs report
//               their bytes to the even CTA's barriers.
//   warp 1      allocates TMEM in both CTAs; in the even CTA it issues every
//               MMA of the pair and commits each completion to the barrier
//               of that name in both CTAs.
//   warps 2..9  softmax, two warps per TMEM lane quadrant that take the key
//               tiles in turn (a whole 128-key row of S each); only the
//               running row maximum passes from one to the other, so the two
//               warps, which share a scheduler, run half a tile apart.  P
//               (bf16) is written over the first 64 columns of the S buffer.
//               The same warps rescale O (when a row maximum grew by more
//               than 2^8) and run the epilogue, 64 columns each.
// Every output row is computed by one CTA in a fixed key-tile order that
// depends only on its own sequence, so results do not depend on the rest of
// the batch.  Key columns past the sequence end are masked to -inf (P = 0)
// and V rows past it are cleared in shared memory (0 * NaN would be NaN);
// query rows past it are computed but never stored.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"
#include "tma_map.h"
#include "varlen_items.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTile = kVarlenTile;          // query rows per CTA, keys per key tile
constexpr int kItemRows = kVarlenItemRows;  // query rows per work item (one pair)
constexpr int kCluster = 2;
constexpr int kSBufs = 3;           // S/P buffers in TMEM
constexpr int kThreads = 320;       // producer, MMA issuer, 8 softmax warps
constexpr int kQBufs = 2;           // Q tile buffers
constexpr int kSlots = 9;           // K/V ring slots
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;  // teardown after an abort (~0.2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units

struct PairCfg {
  static constexpr int kHalfBytes = kTile * 128;    // 128 rows x 128 B (64 columns)
  static constexpr int kQBytes = 2 * kHalfBytes;    // one 128 x 128 Q tile
  static constexpr int kKHalfBytes = 64 * 128;      // 64 keys x 128 B
  static constexpr int kSlotBytes = 16384;          // a K half-tile or a V half-tile
  static constexpr int kQOff = 0;                   // kQBufs Q buffers
  static constexpr int kRingOff = kQBufs * kQBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
  static constexpr int kQFull = 0,      // [kQBufs] even CTA: Q bytes of both CTAs
      kQEmpty = 2,                      // [kQBufs] both: the item's last S is done
      kSFull = 4,                       // [3] both: S of a key tile is done
      kPReady = 7,                      // [3] even CTA: the pair's 8 warps of the tile wrote P
      kOFull = 10,                      // both: the item's last PV is done
      kFinal = 11,                      // even CTA: every MMA done (teardown)
      kTail = 12,                       // own: a V half-tile whose tail rows are cleared
      kSlotFull = 13,                   // [kSlots] even CTA: both CTAs' bytes
      kSlotEmpty = 13 + kSlots;         // [kSlots] both
  static constexpr int kNumBars = 13 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag
  // softmax hand-off: running row maxima [quadrant][to side][lane] and
  // their ok flags [quadrant][to side]; epilogue (sum, its maximum) pairs
  // [item parity][quadrant][side][lane] and ok flags [item parity][quadrant][side]
  static constexpr int kXMaxOff = (kMiscOff + 16 + 127) / 128 * 128;
  static constexpr int kXOkOff = kXMaxOff + 4 * 2 * 32 * 4;
  static constexpr int kXSumOff = kXOkOff + 4 * 2 * 4;
  static constexpr int kXSumOkOff = kXSumOff + 2 * 4 * 2 * 32 * 8;
  static constexpr int kSchedOff = (kXSumOkOff + 2 * 4 * 2 * 4 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kSchedOff + (2 * PA_MAX_BATCH + 1) * 4;
  static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-CTA limit");
  static constexpr uint32_t kColO = kSBufs * kTile;  // S buffers at 0, 128, 256
  static constexpr uint32_t kTmemCols = 512;
  // K-major Q and K; V MN-major; M spans the pair
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kCluster * kTile, kTile, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kCluster * kTile, kD, true);
};

// A position in a pair's stream of key tiles: items i0, i0 + stride, ...,
// skipping items without keys; tile j of item i.  done() once past the end.
struct Walk {
  int i, j, n_items, stride;
  ItemInfo it;
  __device__ __forceinline__ bool done() const { return i >= n_items; }
};
__device__ __forceinline__ void walk_seek(Walk &w, const VarlenParams &p, const int32_t *order,
                                          const int32_t *prefix) {
  w.j = 0;
  while (w.i < w.n_items) {
    w.it = item_info(p, order, prefix, w.i);
    if (w.it.nk > 0) return;
    w.i += w.stride;
  }
}
__device__ __forceinline__ void walk_next(Walk &w, const VarlenParams &p, const int32_t *order,
                                          const int32_t *prefix) {
  if (++w.j < w.it.nk) return;
  w.i += w.stride;
  walk_seek(w, p, order, prefix);
}

// Row maximum of 128 raw scores (TMEM words), over the first `valid` keys;
// with a positive scale the maximum of the raw scores is scaled once,
// otherwise every score is scaled first.  The unmasked positive-scale form
// (every tile but a sequence's last) is three-input max chains only.
__device__ __forceinline__ float tile_max(const uint32_t (&sr)[kTile], int valid, float sl2) {
  float mx8[8];
  if (sl2 > 0.f && valid >= kTile) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      mx8[e] = fmaxf(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
#pragma unroll
    for (int c = 8; c < kTile / 2; ++c)
      mx8[c & 7] = fmax3(mx8[c & 7], __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
    for (int c = 0; c < kTile; ++c) {
      float v = __uint_as_float(sr[c]);
      if (!(sl2 > 0.f)) v *= sl2;
      if (c >= valid) v = -INFINITY;
      mx8[c & 7] = fmaxf(mx8[c & 7], v);
    }
  }
  const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                         fmaxf(mx8[6], mx8[7]));
  return sl2 > 0.f ? mx * sl2 : mx;
}

// P = 2^(s * scale_log2 - m) for the 128 keys of one TMEM lane's S row at
// `taddr`, 64 at a time, written as bf16 pairs over the row's first 64
// columns; adds P to the eight partial sums.  kMasked: keys from `valid` on
// get P = 0 (a sequence's last key tile).
template <bool kMasked>
__device__ __forceinline__ void tile_p(uint32_t taddr, int valid, float sl2, float m,
                                       float2 (&sum8)[8]) {
  const float2 sl22 = make_float2(sl2, sl2), negm2 = make_float2(-m, -m);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t sr[64];
    tmem_ld32(taddr + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_ld32(taddr + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_wait_ld();
    uint32_t pk[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float2 tt = __ffma2_rn(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                             sl22, negm2);
      if (kMasked) {
        if (hh * 64 + 2 * c >= valid) tt.x = -INFINITY;
        if (hh * 64 + 2 * c + 1 >= valid) tt.y = -INFINITY;
      }
      const float2 pp = make_float2(ex2(tt.x), ex2(tt.y));
      sum8[c & 7] = __fadd2_rn(sum8[c & 7], pp);
      pk[c] = pack_bf16x2(pp.x, pp.y);
    }
    tmem_st32(taddr + hh * 32, pk);
  }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    varlen_attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const VarlenParams p) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need a 1024-byte aligned base.  Both CTAs of a
  // pair run the same code on the same layout, so both skip or neither.
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) record_error(p.status, PA_DEVICE_ERR_SMEM_ALIGN);
    return;
  }
  uint8_t *gbase = smem_raw;
  const uint32_t sQ = base + C::kQOff;
  const uint32_t sRing = base + C::kRingOff;
  auto bar = [&](int idx) -> uint32_t { return base + C::kBarOff + 8u * idx; };
  uint32_t *tmem_base_ptr = reinterpret_cast<uint32_t *>(gbase + C::kMiscOff);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(gbase + C::kMiscOff + 4);
  int32_t *order = reinterpret_cast<int32_t *>(gbase + C::kSchedOff);
  int32_t *prefix = order + PA_MAX_BATCH;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  // ---- set-up: barriers, TMEM, work list --------------------------------
  if (tid == 0) {
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(bar(C::kQFull + b), 1);    // the even CTA's expect_tx; bytes of both CTAs
      mbar_init(bar(C::kQEmpty + b), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPReady + b), 4 * kCluster);   // the tile's softmax warps in the pair
    }
    mbar_init(bar(C::kOFull), 1);
    mbar_init(bar(C::kFinal), 1);
    mbar_init(bar(C::kTail), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(C::kSlotFull + s), 1);   // as kQFull
      mbar_init(bar(C::kSlotEmpty + s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(base + C::kMiscOff, C::kTmemCols);
  // the ring is free until the first load: use it for the build's temporaries
  int32_t *tmp = reinterpret_cast<int32_t *>(gbase + C::kRingOff);
  sched_build(order, prefix, tmp, tmp + PA_MAX_BATCH, p.cu_q, p.cu_k, p.batch, p.H, kItemRows,
              p.total_q, p.total_k, p.max_q, p.max_k, p.status, blockIdx.x == 0);
  fence_before_sync();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();   // barriers of both CTAs initialised before any remote use
  fence_after_sync();
  const uint32_t tmem = *tmem_base_ptr;
  const int n_items = prefix[p.batch];
  const int cl = blockIdx.x / kCluster, n_cl = gridDim.x / kCluster;

  if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
    const bool lead = elect_one();
    if (lead) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t loads = 0, q_loads = 0, tails = 0;
    bool ok = true, tail_pending = false;
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = bounded_wait_cluster(b, parity, abort_flag, p.status, kWaitLimit);
      return __all_sync(0xffffffffu, w);
    };
    // next ring slot in load order, once the MMAs that read it are done
    auto take_slot = [&](uint32_t &s) -> bool {
      s = loads % kSlots;
      return wait_all(bar(C::kSlotEmpty + s), ((loads / kSlots) & 1u) ^ 1u);
    };
    auto load_q = [&](const ItemInfo &it) -> bool {
      const uint32_t qb = q_loads % kQBufs;
      if (!wait_all(bar(C::kQEmpty + qb), ((q_loads / kQBufs) & 1u) ^ 1u)) return false;
      if (lead) {
        const uint32_t full = mapa_shared(bar(C::kQFull + qb), 0);
        if (leader) mbar_arrive_expect_tx(bar(C::kQFull + qb), kCluster * C::kQBytes);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d_pair(sQ + qb * C::kQBytes + hf * C::kHalfBytes, &tm_q, full, hf * 64,
                           it.head, it.q_row0 + static_cast<int>(rank) * kTile);
      }
      ++q_loads;
      return true;
    };
    // this CTA's 64 keys of the K tile, all 128 columns
    auto load_k = [&](const Walk &w) -> bool {
      uint32_t s;
      if (!take_slot(s)) return false;
      const int row = w.it.k0 + key_tile(w.it, w.j) * kTile + static_cast<int>(rank) * 64;
      if (lead) {
        const uint32_t full = mapa_shared(bar(C::kSlotFull + s), 0);
        if (leader) mbar_arrive_expect_tx(bar(C::kSlotFull + s), kCluster * C::kSlotBytes);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d_pair(sRing + s * C::kSlotBytes + hf * C::kKHalfBytes, &tm_k, full,
                           hf * 64, w.it.head, row);
      }
      ++loads;
      return true;
    };
    // this CTA's 64 columns of the V tile, all 128 keys
    auto load_v = [&](const Walk &w) -> bool {
      uint32_t s;
      if (!take_slot(s)) return false;
      const int kt = key_tile(w.it, w.j);
      const int row = w.it.k0 + kt * kTile;
      const int valid = w.it.lk - kt * kTile;
      const uint32_t dst = sRing + s * C::kSlotBytes;
      const uint32_t full = mapa_shared(bar(C::kSlotFull + s), 0);
      if (lead && leader) mbar_arrive_expect_tx(bar(C::kSlotFull + s), kCluster * C::kSlotBytes);
      if (valid >= kTile) {
        if (lead) tma_load_3d_pair(dst, &tm_v, full, static_cast<int>(rank) * 64, w.it.head, row);
      } else {
        // The tile holds rows past the sequence end (the next sequence's, or
        // the buffer's trailing rows).  P is 0 there, but 0 * Inf and
        // 0 * NaN are NaN, so those rows are zeroed before the MMAs may read
        // the slot: the copy completes on this CTA's own barrier, the rows
        // are cleared, and only then are its bytes counted on the slot.
        if (lead) {
          mbar_arrive_expect_tx(bar(C::kTail), C::kSlotBytes);
          tma_load_3d(dst, &tm_v, bar(C::kTail), static_cast<int>(rank) * 64, w.it.head, row);
        }
        tail_pending = true;
        if (!wait_all(bar(C::kTail), tails & 1u)) return false;
        tail_pending = false;
        ++tails;
        // one 64-column half: 128 rows x 128 B; the 128-byte swizzle only
        // permutes 16-byte chunks inside a row, so whole rows are cleared
        // without unswizzling.  The proxy fences order the stores after the
        // TMA bytes and before the tensor core's reads (both async-proxy);
        // the release fence publishes them to the even CTA's MMA issuer.
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        uint8_t *tile = gbase + C::kRingOff + s * C::kSlotBytes;
        for (int c = lane; c < (kTile - valid) * 8; c += 32)
          *reinterpret_cast<uint4 *>(tile + (valid + (c >> 3)) * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        fence_acq_rel_cluster();
        __syncwarp();
        if (lead) mbar_complete_tx_remote(full, C::kSlotBytes);
      }
      ++loads;
      return true;
    };
    Walk kw{cl, 0, n_items, n_cl, {}}, vw{cl, 0, n_items, n_cl, {}};
    walk_seek(kw, p, order, prefix);
    walk_seek(vw, p, order, prefix);
    // the order of the MMA issuer: K of the first kSBufs tiles, then V_g, K_{g+3}
    auto next_k = [&]() -> bool {
      if (kw.done()) return true;
      if (kw.j == 0 && !load_q(kw.it)) return false;
      if (!load_k(kw)) return false;
      walk_next(kw, p, order, prefix);
      return true;
    };
    for (int t = 0; t < kSBufs && ok; ++t) ok = next_k();
    while (ok && !vw.done()) {
      ok = load_v(vw);
      walk_next(vw, p, order, prefix);
      if (ok) ok = next_k();
    }
    if (!ok) {
      // give the copies already issued a bounded chance to land (the even
      // CTA's barriers count both CTAs' bytes)
      if (leader) {
        for (uint32_t s = 0; s < static_cast<uint32_t>(kSlots) && s < loads; ++s) {
          const uint32_t n = (loads - s + kSlots - 1) / kSlots;  // loads into slot s
          drain_wait(bar(C::kSlotFull + s), (n - 1) & 1u, kDrainLimit);
        }
        for (uint32_t b = 0; b < static_cast<uint32_t>(kQBufs) && b < q_loads; ++b) {
          const uint32_t n = (q_loads - b + kQBufs - 1) / kQBufs;   // loads into buffer b
          drain_wait(bar(C::kQFull + b), (n - 1) & 1u, kDrainLimit);
        }
      }
      if (tail_pending) drain_wait(bar(C::kTail), tails & 1u, kDrainLimit);
    }
  } else if (warp == 1) {
    // ================= MMA issuer (the even CTA only) =================
    // Issue order over the pair's stream of key tiles g (across items):
    //   S_0 S_1 S_2 | PV_0 S_3 | PV_1 S_4 | ...
    // S_g goes to S buffer g % 3; S_{g+3} is issued after PV_g, which reads
    // P_g from that buffer, and one thread's MMAs execute in order.  Past
    // the stream's end a commit without an MMA keeps the S_full phases
    // counting, so "S_full of index g + 2 done" always means "PV_{g-1}
    // done" (the softmax's O-rescale wait).
    // The whole warp runs the issuer (warp-uniform operands); one elected
    // lane issues each MMA and commit.
    if (leader) {
      const bool lead = elect_one();
      auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
        const bool w = bounded_wait_cluster(b, parity, abort_flag, p.status, kWaitLimit);
        return __all_sync(0xffffffffu, w);
      };
      // commit to the same barrier in both CTAs of the pair
      auto commit_both = [&](uint32_t b) {
        if (lead) {
          mma_commit_pair(mapa_shared(b, 0));
          mma_commit_pair(mapa_shared(b, 1));
        }
      };
      uint32_t slot_uses = 0, kq = 0, gs = 0, gv = 0;
      bool ok = true, issued = false;
      auto next_slot = [&](uint32_t &s) -> bool {
        s = slot_uses % kSlots;
        const bool r = wait_all(bar(C::kSlotFull + s), (slot_uses / kSlots) & 1u);
        ++slot_uses;
        return r;
      };
      // descriptors advance by adding the byte offset >> 4 to the start
      // address field; every operand lies below 256 KB, so nothing carries
      const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(sRing, 16, 1024);
      // V (MN-major): one 64-column half per CTA, next 8 keys at SBO = 1024
      const uint64_t vdesc0 = sdesc_sw128(sRing, 1024, 1024);
      Walk kw{cl, 0, n_items, n_cl, {}}, vw{cl, 0, n_items, n_cl, {}};
      walk_seek(kw, p, order, prefix);
      walk_seek(vw, p, order, prefix);
      // S_gs = Q K^T of the K walk's tile (or a bare commit past the end)
      auto issue_s = [&]() -> bool {
        const uint32_t b = gs % kSBufs;
        if (kw.done()) {
          commit_both(bar(C::kSFull + b));
          ++gs;
          return true;
        }
        const uint32_t qb = kq % kQBufs;
        if (kw.j == 0 && !wait_all(bar(C::kQFull + qb), (kq / kQBufs) & 1u)) return false;
        uint32_t s;
        if (!next_slot(s)) return false;
        const uint64_t a0 = qdesc0 + ((qb * C::kQBytes) >> 4);
        const uint64_t b0 = kdesc0 + ((s * C::kSlotBytes) >> 4);
        const uint32_t d_s = tmem + b * kTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t oa = ((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * C::kKHalfBytes + (kk & 3) * 32) >> 4;
          if (lead) mma_ss_pair(d_s, a0 + oa, b0 + ob, C::kIdescS, kk > 0 ? 1u : 0u);
        }
        issued = true;
        commit_both(bar(C::kSFull + b));
        commit_both(bar(C::kSlotEmpty + s));
        if (kw.j == kw.it.nk - 1) {   // the item's last S: its Q buffer is free
          commit_both(bar(C::kQEmpty + qb));
          ++kq;
        }
        ++gs;
        walk_next(kw, p, order, prefix);
        return true;
      };
      if (!vw.done())
        for (int t = 0; t < kSBufs && ok; ++t) ok = issue_s();
      while (ok && !vw.done()) {
        const uint32_t b = gv % kSBufs;
        // P_gv written by the pair's 16 softmax warps
        if (!wait_all(bar(C::kPReady + b), (gv / kSBufs) & 1u)) {
          ok = false;
          break;
        }
        fence_after_sync();
        uint32_t s;
        if (!next_slot(s)) {
          ok = false;
          break;
        }
        // O += P V (P, bf16, over the first 64 columns of the S buffer)
        const uint64_t b0 = vdesc0 + ((s * C::kSlotBytes) >> 4);
        const uint32_t d_p = tmem + b * kTile;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (lead)
            mma_ts_pair(tmem + C::kColO, d_p + kk * 8, b0 + ((kk * 16 * 128) >> 4), C::kIdescO,
                        (vw.j == 0 && kk == 0) ? 0u : 1u);
        }
        issued = true;
        if (vw.j == vw.it.nk - 1) commit_both(bar(C::kOFull));
        commit_both(bar(C::kSlotEmpty + s));
        ++gv;
        walk_next(vw, p, order, prefix);
        ok = issue_s();
      }
      // every MMA issued so far has finished before TMEM is released
      if (issued) {
        if (lead) mma_commit_pair(mapa_shared(bar(C::kFinal), 0));
        drain_wait(bar(C::kFinal), 0, kWaitLimit);
      }
    }
    __syncwarp();
  } else {
    // ================= softmax / rescale / epilogue =================
    // The two warps of a TMEM lane quadrant (warp % 4, a hardware rule) take
    // the stream's key tiles in turn: warps 2..5 the even tiles g, warps
    // 6..9 the odd ones, each a whole 128-key row of S.  Only the running row
    // maximum passes from a tile's warp to the next tile's, through shared
    // memory and a named barrier that the writer arrives on without waiting,
    // so the two warps (which share a scheduler) run half a tile apart.
    // Each warp sums P over its own tiles; the two sums meet in the epilogue.
    const int quad = warp & 3;
    const int side = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t p_ready0 = mapa_shared(bar(C::kPReady), 0);
    float *xm = reinterpret_cast<float *>(gbase + C::kXMaxOff);          // [quad][to side][lane]
    int32_t *xok = reinterpret_cast<int32_t *>(gbase + C::kXOkOff);     // [quad][to side]
    float *xs = reinterpret_cast<float *>(gbase + C::kXSumOff);         // [item parity][quad][side][lane][2]
    int32_t *xs_ok = reinterpret_cast<int32_t *>(gbase + C::kXSumOkOff);  // [item parity][quad][side]
    const int to_me = quad * 2 + side, to_other = quad * 2 + (side ^ 1);
    const float sl2 = p.scale_log2;
    uint32_t g = 0, o_waits = 0;
    bool ok = true;
    for (int i = cl; i < n_items && ok; i += n_cl) {
      const ItemInfo it = item_info(p, order, prefix, i);
      const int rows_c = it.rows - static_cast<int>(rank) * kTile;   // may be <= 0
      __nv_bfloat16 *dst =
          p.out +
          (static_cast<int64_t>(it.q_row0 + static_cast<int>(rank) * kTile + row) * p.H +
           it.head) * kD + side * 64;
      const bool store = row < rows_c;
      if (it.nk == 0) {
        if (store) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
          for (int c = 0; c < 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // m: running maximum after this warp's latest tile; l: this warp's P
      // sum, scaled to m_ref
      float m = -INFINITY, l = 0.f, m_ref = -INFINITY;
      for (int j = 0; j < it.nk && ok; ++j, ++g) {
        if (static_cast<int>(g & 1u) != side) continue;
        const uint32_t b = g % kSBufs;
        bool okt = bounded_wait_cluster(bar(C::kSFull + b), (g / kSBufs) & 1u, abort_flag,
                                        p.status, kWaitLimit);
        okt = __all_sync(0xffffffffu, okt);
        // pass 1: the tile's row maximum (scores are read again for P, so
        // no 128-value array stays live across the hand-off)
        const int valid = key_tile(it, j) == it.nk - 1 ? it.lk - (it.nk - 1) * kTile : kTile;
        float mx = -INFINITY;
        if (okt) {
          fence_after_sync();
          uint32_t sr[kTile];
#pragma unroll
          for (int c = 0; c < kTile / 32; ++c)
            tmem_ld32(lane_base + b * kTile + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
          tmem_wait_ld();
          mx = tile_max(sr, valid, sl2);
        }
        // the running maximum after the previous tile (the other warp's)
        float m_prev = -INFINITY;
        if (j > 0) {
          named_bar_sync(1 + to_me, 64);
          m_prev = xm[to_me * 32 + lane];
          if (xok[to_me] == 0) okt = false;
        }
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = mx;
        } else if (mx > m_prev + kRescaleThreshold) {
          alpha = ex2(m_prev - mx);
          m = mx;
          rescale = true;
        } else {
          m = m_prev;
        }
        const bool any_rescale = okt && __any_sync(0xffffffffu, rescale);
        if (any_rescale) {
          // O must hold PV_{g-1}: S of index g + 2 is issued right after it
          // (or a bare commit past the stream's end)
          const bool w2 = bounded_wait_cluster(bar(C::kSFull + (g + 2) % kSBufs),
                                               ((g + 2) / kSBufs) & 1u, abort_flag, p.status,
                                               kWaitLimit);
          okt = __all_sync(0xffffffffu, w2);
        }
        // hand the running maximum (and whether this warp goes on) to the
        // next tile's warp; the barrier is left without waiting
        if (j + 1 < it.nk) {
          xm[to_other * 32 + lane] = m;
          if (lane == 0) xok[to_other] = okt ? 1 : 0;
          named_bar_arrive(1 + to_other, 64);
        }
        if (!okt) {
          ok = false;
          break;
        }
        // pass 2: P as bf16 over the first 64 columns of the S buffer
        float2 sum8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sum8[e] = make_float2(0.f, 0.f);
        if (valid >= kTile)
          tile_p<false>(lane_base + b * kTile, valid, sl2, m, sum8);
        else
          tile_p<true>(lane_base + b * kTile, valid, sl2, m, sum8);
        const float2 s01 = __fadd2_rn(__fadd2_rn(sum8[0], sum8[1]), __fadd2_rn(sum8[2], sum8[3]));
        const float2 s45 = __fadd2_rn(__fadd2_rn(sum8[4], sum8[5]), __fadd2_rn(sum8[6], sum8[7]));
        const float2 s8 = __fadd2_rn(s01, s45);
        if (m != m_ref) {   // bring this warp's earlier sum to the current maximum
          l *= ex2(m_ref - m);
          m_ref = m;
        }
        l += s8.x + s8.y;
        // rescale O in place (PV_{g-1} is done, PV_g waits for this warp)
        if (any_rescale) {
          fence_after_sync();
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + C::kColO + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(lane_base + C::kColO + c * 32, r);
          }
        }
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(p_ready0 + 8u * b);
      }
      // epilogue: wait for the item's last PV, combine the two warps' sums,
      // normalise this warp's 64 columns of O and store the valid rows.  The
      // exchange runs even after a failure, so both warps stop together.
      bool oko = ok;
      if (oko) {
        oko = bounded_wait_cluster(bar(C::kOFull), o_waits & 1u, abort_flag, p.status,
                                   kWaitLimit);
        oko = __all_sync(0xffffffffu, oko);
      }
      const int par = static_cast<int>(o_waits & 1u) * 8;
      ++o_waits;
      xs[((par + to_me) * 32 + lane) * 2 + 0] = l;
      xs[((par + to_me) * 32 + lane) * 2 + 1] = m_ref;
      if (lane == 0) xs_ok[par + to_me] = oko ? 1 : 0;
      named_bar_sync(9 + quad, 64);
      if (!oko || xs_ok[par + to_other] == 0) {
        ok = false;
        break;
      }
      const float l_o = xs[((par + to_other) * 32 + lane) * 2 + 0];
      const float m_o = xs[((par + to_other) * 32 + lane) * 2 + 1];
      const float m_fin = fmaxf(m_ref, m_o);   // the maximum after the item's last tile
      const float inv = 1.f / (l * ex2(m_ref - m_fin) + l_o * ex2(m_o - m_fin));
      fence_after_sync();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColO + side * 64 + c * 32, r);
        tmem_wait_ld();
        if (store) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
            d4[v] = w;
          }
        }
      }
    }
  }

  // ---- teardown -------------------------------------------------------------
  // neither CTA leaves while the other may still read its shared memory,
  // arrive on its barriers or run MMAs on its TMEM
  fence_before_sync();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();
  fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// [rows, H, 128] bf16 viewed as a 3-D tensor (D, H, rows); box 64 x 1 x
// box_rows with 128-byte swizzle.  Rows past the end read as zero.
bool make_map_rows(CUtensorMap *map, const void *ptr, int rows, int H, int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(H) * kD * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_varlen_attn_pair(const VarlenArgs &a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map_rows(&mq, a.q, a.total_q, a.H, kTile) ||
      !make_map_rows(&mk, a.k, a.total_k, a.H, 64) ||
      !make_map_rows(&mv, a.v, a.total_k, a.H, kTile))
    return cudaErrorInvalidValue;
  VarlenParams p;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.batch = a.batch;
  p.H = a.H;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.max_q = a.max_q;
  p.max_k = a.max_k;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(varlen_attn_pair_kernel),
                                PairCfg::kSmemBytes, configured);
  if (e != cudaSuccess) return e;
  const int grid = a.num_sms / kCluster * kCluster;   // whole pairs, one CTA per SM
  varlen_attn_pair_kernel<<<grid, kThreads, PairCfg::kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace pa
