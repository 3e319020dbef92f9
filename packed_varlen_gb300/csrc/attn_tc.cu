// Packed variable-length attention on the 5th-generation tensor cores.
//
// Computes, per sequence b, head h and query row i of b, softmax attention
// over the key rows of the same sequence only (the flat varlen path of
// "[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
// varlen attention for mixfusion", Key changes; "feat: Support dynamic
// batching for heterogeneous diffusion requests", AttentionMetadata).
//
// This kernel serves head dim 64; head dim 128 runs on the CTA-pair kernel
// (attn_pair.cu), whose M = 256 MMAs leave TMEM room to compute scores
// ahead of the softmax.
//
// Design: one persistent CTA per SM, 11 warps.  A work item is 256 query
// rows of one (sequence, head), held as two 128-row tiles Q0 and Q1 that share
// every K/V tile loaded, so each K/V byte brought into shared memory feeds
// twice the tensor-core work of a single-tile item.
//   warp 0      TMA producer: Q0/Q1 once per item, then K0, V0, K1, V1, ...
//               through a ring of shared-memory slots.
//   warp 1      allocates TMEM (S0, S1, O0, O1: 128 columns each) and
//               issues tile 0's tcgen05.mma in the order
//                 S0_0 | PV0_0 S0_1 | PV0_1 S0_2 ...
//   warp 10     issues tile 1's in the same order.
//               S = Q K^T with both operands in shared memory, fp32 into TMEM;
//               O += P V with P (bf16) read from TMEM, V from shared memory.
//               While one tile's softmax runs, the tensor core computes the
//               other tile's PV and next S.  Each issuer is a whole warp
//               with one elected lane issuing (warp-uniform operands), and
//               the two take turns group by group; with two issuers one
//               thread's waits, fences and commits overlap the other's MMAs.
//   warps 2..5  softmax of tile 0, one thread per query row (TMEM lane);
//   warps 6..9  softmax of tile 1.  Each thread reads its row of S, runs the
//               online softmax in fp32 (exp2 with the scale folded in),
//               writes P as bf16 over the first 64 columns of its S buffer,
//               rescales O in TMEM only when the row maximum grew by more
//               than 2^8, and finally normalises O and stores bf16 rows.
// P overwrites S in place: the MMA that next writes that S buffer is issued
// after the PV that reads P by the same thread, and one thread's tcgen05
// MMAs execute in order.
// Every output row is computed by one CTA in a fixed key-tile order that
// depends only on its own sequence, so results do not depend on the rest of
// the batch.  Key columns past the sequence end are masked to -inf (P = 0);
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

constexpr int kTile = kVarlenTile;          // rows of a Q tile, keys of a K/V tile
constexpr int kItemRows = kVarlenItemRows;  // query rows per work item (two tiles)
constexpr int kThreads = 352;       // producer, 2 MMA issuers, 2 x 4 softmax warps
constexpr int kMmaWarp1 = kThreads / 32 - 1;   // issuer of tile 1
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;  // teardown after an abort (~0.2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units

// Shared-memory plan for head dim D, kSlots K/V ring slots and a work list
// of up to kMaxSeqs sequences.  The dynamic shared-memory window starts
// 1024-byte aligned (checked at run time), so no alignment slack is added.
template <int D, int kSlots_, int kMaxSeqs_>
struct Cfg {
  static constexpr int kSlots = kSlots_;
  static constexpr int kMaxSeqs = kMaxSeqs_;
  static constexpr int kHalfBytes = kTile * 64 * 2;         // 128 rows x 128 B
  static constexpr int kTileBytes = kTile * D * 2;          // one Q/K/V tile
  static constexpr int kQOff = 0;                           // Q0, Q1
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // barriers: per Q tile t an S-full, a P-ready and an O-full barrier
  static constexpr int kQFull = 0, kQEmpty = 1, kSFull = 2, kPReady = 4, kOFull = 6,
                       kFinal = 8, kTurn = 10, kSlotFull = 12, kSlotEmpty = 12 + kSlots;
  static constexpr int kNumBars = 12 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kSchedOff = (kMiscOff + 16 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kSchedOff + (2 * kMaxSeqs + 1) * 4;
  static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-CTA limit");
  // TMEM columns: S_t at 128 t (P_t over its first 64), O_t at 256 + D t
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, kTile, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kTile, D, true);
  // V (MN-major): next 64-column half at LBO, next 8 keys at SBO = 1024.  With
  // D = 64 the MMA spans a single half and LBO is never used.
  static constexpr uint32_t kVLbo = D == 128 ? kHalfBytes : 1024;
};

// Whole warp: zero key rows [valid, 128) of a V tile in shared memory.  The
// tile is D / 64 column halves of 128 rows x 128 bytes; the 128-byte swizzle
// only permutes the 16-byte chunks inside a row, so a whole row is cleared
// without unswizzling.  The fences order the stores after the TMA bytes that
// landed and before the tensor core's reads (both are async-proxy accesses).
template <int D>
__device__ __forceinline__ void zero_v_tail(uint8_t *tile, int valid, int lane) {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  const int per_half = (kTile - valid) * 8;   // 16-byte chunks per half
  for (int c = lane; c < per_half * (D / 64); c += 32) {
    const int hf = c / per_half, r = c - hf * per_half;
    *reinterpret_cast<uint4 *>(tile + hf * (kTile * 128) + (valid + (r >> 3)) * 128 +
                               (r & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  __syncwarp();
}

template <int D, int kSlots, int kMaxSeqs>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const VarlenParams p) {
  using C = Cfg<D, kSlots, kMaxSeqs>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need a 1024-byte aligned base
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
  int32_t *prefix = order + kMaxSeqs;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- set-up: barriers, TMEM, work list --------------------------------
  if (tid == 0) {
    mbar_init(bar(C::kQFull), 1);
    mbar_init(bar(C::kQEmpty), 2);   // one arrival per MMA issuer
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kSFull + t), 1);
      mbar_init(bar(C::kPReady + t), 128);
      mbar_init(bar(C::kOFull + t), 1);
    }
    mbar_init(bar(C::kFinal + 0), 1);
    mbar_init(bar(C::kFinal + 1), 1);
    mbar_init(bar(C::kTurn + 0), 1);
    mbar_init(bar(C::kTurn + 1), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kSlotFull + s), 1);
      mbar_init(bar(C::kSlotEmpty + s), 2);   // one arrival per MMA issuer
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(base + C::kMiscOff, C::kTmemCols);
  // the ring is free until the first load: use it for the build's temporaries
  int32_t *tmp = reinterpret_cast<int32_t *>(gbase + C::kRingOff);
  sched_build(order, prefix, tmp, tmp + kMaxSeqs, p.cu_q, p.cu_k, p.batch, p.H,
              kItemRows, p.total_q, p.total_k, p.max_q, p.max_k, p.status, blockIdx.x == 0);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_base_ptr;
  const int n_items = prefix[p.batch];

  if (warp == 0) {
    // ================= TMA producer =================
    // (warp-wide like the MMA issuers: one elected lane issues the copies)
    {
      const bool lead = elect_one();
      if (lead) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      uint32_t q_loads = 0, slot_loads = 0;
      bool ok = true;
      auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
        const bool w = bounded_wait(b, parity, abort_flag, p.status, kWaitLimit);
        return __all_sync(0xffffffffu, w);
      };
      auto load_kv = [&](const CUtensorMap *tm, int row, int head) -> bool {
        const uint32_t s = slot_loads % C::kSlots;
        const uint32_t use = slot_loads / C::kSlots;
        if (!wait_all(bar(C::kSlotEmpty + s), (use & 1u) ^ 1u)) return false;
        const uint32_t dst = sRing + s * C::kTileBytes;
        if (lead) {
          mbar_arrive_expect_tx(bar(C::kSlotFull + s), C::kTileBytes);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_3d(dst + hf * C::kHalfBytes, tm, bar(C::kSlotFull + s), hf * 64, head, row);
        }
        ++slot_loads;
        return true;
      };
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const ItemInfo it = item_info(p, order, prefix, i);
        if (it.nk == 0) continue;
        const int ntq = it.rows > kTile ? 2 : 1;
        if (!wait_all(bar(C::kQEmpty), (q_loads & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        if (lead) {
          mbar_arrive_expect_tx(bar(C::kQFull), ntq * C::kTileBytes);
          for (int t = 0; t < ntq; ++t) {
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              tma_load_3d(sQ + t * C::kTileBytes + hf * C::kHalfBytes, &tm_q, bar(C::kQFull),
                          hf * 64, it.head, it.q_row0 + t * kTile);
          }
        }
        ++q_loads;
        for (int j = 0; j < it.nk && ok; ++j) {
          const int row = it.k0 + key_tile(it, j) * kTile;
          ok = load_kv(&tm_k, row, it.head);
          if (ok) ok = load_kv(&tm_v, row, it.head);
        }
      }
      if (!ok) {
        // give the copies already issued a bounded chance to land
        for (uint32_t s = 0; s < C::kSlots && s < slot_loads; ++s) {
          const uint32_t n = (slot_loads - s + C::kSlots - 1) / C::kSlots;  // loads into s
          drain_wait(bar(C::kSlotFull + s), (n - 1) & 1u, kDrainLimit);
        }
        if (q_loads) drain_wait(bar(C::kQFull), (q_loads - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ================= MMA issuers: warp 1 for tile 0, the last warp for tile 1 ====
    // Each issuer walks the same items and the same ring slots; it issues its
    // own tile's MMAs in the order S_0 | PV_0 S_1 | PV_1 S_2 ... and frees a
    // slot (or the Q buffer) with one arrival on a two-arrival barrier: a
    // commit once its MMAs reading the slot are done, or a plain arrive when
    // its tile is absent from the item.
    // The whole warp runs the issuer, so every operand of an MMA is
    // warp-uniform, and one elected lane issues each MMA, commit and
    // arrive: tcgen05.mma issued from a lone lane's control flow costs about
    // 100 cycles per instruction, against 64 of tensor work for these shapes.
    const int t = warp == 1 ? 0 : 1;
    {
      const bool lead = elect_one();
      uint32_t q_uses = 0, slot_uses = 0, issued = 0, p_waits = 0;
      bool ok = true;
      auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
        const bool w = bounded_wait(b, parity, abort_flag, p.status, kWaitLimit);
        return __all_sync(0xffffffffu, w);
      };
      // next ring slot in consumption order, once its load has landed
      auto wait_slot = [&](uint32_t &s) -> bool {
        s = slot_uses % C::kSlots;
        return wait_all(bar(C::kSlotFull + s), (slot_uses / C::kSlots) & 1u);
      };
      // S_t = Q_t K^T into S buffer t (Q/K K-major, SBO = 8 rows x 128 B)
      // (descriptors advance by adding the byte offset >> 4 to the start
      // address field; every operand lies below 256 KB, so nothing carries)
      const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024) + ((t * C::kTileBytes) >> 4);
      const uint64_t kdesc0 = sdesc_sw128(sRing, 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(sRing, C::kVLbo, 1024);
      const uint32_t d_s = tmem + C::kColS + t * kTile, d_o = tmem + C::kColO + t * D;
      auto issue_s = [&](uint32_t slot) {
        const uint64_t b0 = kdesc0 + ((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4;
          if (lead) mma_ss(d_s, qdesc0 + off, b0 + off, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V (P_t is in the first 64 columns of the S buffer)
      auto issue_pv = [&](uint32_t slot, bool first) {
        const uint64_t b0 = vdesc0 + ((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (lead)
            mma_ts(d_o, d_s + kk * 8, b0 + ((kk * 16 * 128) >> 4), C::kIdescO,
                   (first && kk == 0) ? 0u : 1u);
        }
      };
      // The two issuers take turns group by group (S0_0, S1_0, [PV0_0 S0_1],
      // [PV1_0 S1_1], ...), so the tensor pipe sees the single-thread order
      // that staggers the two tiles; each thread finishes its waits before
      // taking the turn and commits after passing it on.
      uint32_t turns = 0;
      auto take_turn = [&]() -> bool {
        const uint32_t parity = t == 0 ? ((turns & 1u) ^ 1u) : (turns & 1u);
        return wait_all(bar(C::kTurn + t), parity);
      };
      auto pass_turn = [&]() {
        ++turns;
        if (lead) mbar_arrive(bar(C::kTurn + (1 - t)));
      };
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const ItemInfo it = item_info(p, order, prefix, i);
        if (it.nk == 0) continue;
        const bool mine = it.rows > t * kTile;   // this issuer's tile is in the item
        // release a slot / the Q buffer: after this tile's MMAs, or at once
        auto release = [&](uint32_t b) {
          if (!lead) return;
          if (mine)
            mma_commit(b);
          else
            mbar_arrive(b);
        };
        if (!wait_all(bar(C::kQFull), q_uses & 1u)) {
          ok = false;
          break;
        }
        ++q_uses;
        // prologue: S_0 from K_0
        uint32_t sk;
        if (!wait_slot(sk) || !take_turn()) {
          ok = false;
          break;
        }
        if (mine) {
          issue_s(sk);
          issued = 1;
        }
        pass_turn();
        if (mine && lead) mma_commit(bar(C::kSFull + t));
        release(bar(C::kSlotEmpty + sk));
        ++slot_uses;
        if (it.nk == 1) release(bar(C::kQEmpty));
        for (int j = 0; j < it.nk && ok; ++j) {
          const bool more = j + 1 < it.nk;
          uint32_t sv, sk2 = 0;
          if (!wait_slot(sv)) {
            ok = false;
            break;
          }
          ++slot_uses;
          // The last key tile of a sequence whose length is not a multiple
          // of 128 holds rows past the sequence end (the next sequence's, or
          // the buffer's trailing rows).  P is 0 there, but 0 * Inf and
          // 0 * NaN are NaN, so those V rows are zeroed before any PV reads
          // the slot.  Tile 0's issuer runs for every item and issues its PV
          // before tile 1's (the turn order), so it alone clears the rows.
          if (t == 0 && key_tile(it, j) == it.nk - 1) {
            const int valid = it.lk - (it.nk - 1) * kTile;
            if (valid < kTile)
              zero_v_tail<D>(gbase + C::kRingOff + sv * C::kTileBytes, valid, lane);
          }
          if (more && !wait_slot(sk2)) {
            ok = false;
            break;
          }
          // the issue turn first (the order is fixed, so holding it early
          // blocks nobody), then P_j written by this tile's softmax
          if (!take_turn()) {
            ok = false;
            break;
          }
          if (mine) {
            if (!wait_all(bar(C::kPReady + t), p_waits & 1u)) {
              ok = false;
              break;
            }
            ++p_waits;
            fence_after_sync();
          }
          // PV_j, then S_{j+1} (after the PV that reads P from the S buffer)
          if (mine) {
            issue_pv(sv, j == 0);
            if (more) issue_s(sk2);
          }
          pass_turn();
          if (mine && lead) {
            if (more)
              mma_commit(bar(C::kSFull + t));
            else
              mma_commit(bar(C::kOFull + t));
          }
          release(bar(C::kSlotEmpty + sv));
          if (more) {
            release(bar(C::kSlotEmpty + sk2));
            ++slot_uses;
            if (j + 2 == it.nk) release(bar(C::kQEmpty));
          }
        }
      }
      // every MMA this thread issued has finished before TMEM is released
      if (issued) {
        if (lead) mma_commit(bar(C::kFinal + t));
        drain_wait(bar(C::kFinal + t), 0, kWaitLimit);
      }
    }
    __syncwarp();
  } else {
    // ================= softmax / correction / epilogue =================
    // warps 2..5: tile 0, warps 6..9: tile 1; TMEM lane quadrant = warp % 4
    const int t = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t colS = C::kColS + t * kTile;
    const uint32_t colO = C::kColO + t * D;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? sl2 : 1.f;
    uint32_t s_waits = 0, o_waits = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      const ItemInfo it = item_info(p, order, prefix, i);
      const int rows_t = it.rows - t * kTile;   // this tile's valid rows (may be <= 0)
      if (rows_t <= 0) continue;                // tile absent: nothing issued for it
      __nv_bfloat16 *dst =
          p.out + (static_cast<int64_t>(it.q_row0 + t * kTile + row) * p.H + it.head) * D;
      const bool store = row < rows_t;
      if (it.nk == 0) {
        if (store) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.nk; ++j) {
        ok = bounded_wait(bar(C::kSFull + t), s_waits & 1u, abort_flag, p.status, kWaitLimit);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ++s_waits;
        fence_after_sync();
        // all four 32-column loads in flight, then one wait
        uint32_t sr[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
          tmem_ld32(lane_base + colS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_wait_ld();
        // x = raw scores as pairs; with a positive scale the scale is folded
        // into the exponent's FFMA, otherwise the scores are scaled first
        float2 x[kTile / 2];
#pragma unroll
        for (int c = 0; c < kTile / 2; ++c)
          x[c] = make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
        if (!pos_scale) {
          const float2 s2 = make_float2(sl2, sl2);
#pragma unroll
          for (int c = 0; c < kTile / 2; ++c) x[c] = __fmul2_rn(x[c], s2);
        }
        if (key_tile(it, j) == it.nk - 1) {
          const int valid = it.lk - (it.nk - 1) * kTile;
#pragma unroll
          for (int c = 0; c < kTile / 2; ++c) {
            if (2 * c >= valid) x[c].x = -INFINITY;
            if (2 * c + 1 >= valid) x[c].y = -INFINITY;
          }
        }
        // row maximum: eight chains of 3-input max, fixed combine
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(x[e].x, x[e].y);
#pragma unroll
        for (int c = 8; c < kTile / 2; ++c) mx8[c & 7] = fmax3(mx8[c & 7], x[c].x, x[c].y);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7])) * mul;
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = mx;
        } else if (mx > m + kRescaleThreshold) {
          alpha = ex2(m - mx);
          m = mx;
          rescale = true;
        }
        const float2 mul2 = make_float2(mul, mul), negm2 = make_float2(-m, -m);
        float2 sum8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sum8[e] = make_float2(0.f, 0.f);
        uint32_t pk[kTile / 2];
#pragma unroll
        for (int c = 0; c < kTile / 2; ++c) {
          const float2 tt = __ffma2_rn(x[c], mul2, negm2);
          const float2 pp = make_float2(ex2(tt.x), ex2(tt.y));
          sum8[c & 7] = __fadd2_rn(sum8[c & 7], pp);
          pk[c] = pack_bf16x2(pp.x, pp.y);
        }
        const float2 s01 = __fadd2_rn(__fadd2_rn(sum8[0], sum8[1]), __fadd2_rn(sum8[2], sum8[3]));
        const float2 s45 = __fadd2_rn(__fadd2_rn(sum8[4], sum8[5]), __fadd2_rn(sum8[6], sum8[7]));
        const float2 s8 = __fadd2_rn(s01, s45);
        l = l * alpha + (s8.x + s8.y);
        // S_j complete implies the PV issued before it is complete: O is
        // current and can be rescaled in place
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + colO + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(lane_base + colO + c * 32, r);
          }
        }
        // P over the first 64 columns of this tile's S buffer
        {
          uint32_t r[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = pk[e];
          tmem_st32(lane_base + colS, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = pk[32 + e];
          tmem_st32(lane_base + colS + 32, r);
        }
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::kPReady + t));
      }
      if (!ok) break;
      // epilogue: wait for this tile's last PV, normalise, store valid rows
      ok = bounded_wait(bar(C::kOFull + t), o_waits & 1u, abort_flag, p.status, kWaitLimit);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      ++o_waits;
      fence_after_sync();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + colO + c * 32, r);
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
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// [rows, H, D] bf16 viewed as a 3-D tensor (D, H, rows); box 64 x 1 x 128
// with 128-byte swizzle: one 128-row, 64-column half tile per load.
bool make_map(CUtensorMap *map, const void *ptr, int rows, int H, int D) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2};
  const cuuint32_t box[3] = {64, 1, kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kSlots, int kMaxSeqs>
cudaError_t launch_tc(const VarlenArgs &a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.total_q, a.H, D) || !make_map(&mk, a.k, a.total_k, a.H, D) ||
      !make_map(&mv, a.v, a.total_k, a.H, D))
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
  const int smem = Cfg<D, kSlots, kMaxSeqs>::kSmemBytes;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(
      reinterpret_cast<const void *>(varlen_attn_tc_kernel<D, kSlots, kMaxSeqs>), smem,
      configured);
  if (e != cudaSuccess) return e;
  varlen_attn_tc_kernel<D, kSlots, kMaxSeqs><<<a.num_sms, kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

// Head dim 128 runs on the CTA-pair kernel; head dim 64 here, with a
// ten-slot K/V ring beside a work list of up to PA_MAX_BATCH sequences.
cudaError_t launch_varlen_attn(const VarlenArgs &a, cudaStream_t stream) {
  if (a.D == 128) return launch_varlen_attn_pair(a, stream);
  return launch_tc<64, 10, PA_MAX_BATCH>(a, stream);
}

}  // namespace pa
