// Packed variable-length attention on the 5th-generation tensor cores.
//
// Computes, per sequence b, head h and query row i of b, softmax attention
// over the key rows of the same sequence only (the flat varlen path of
// "[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
// varlen attention for mixfusion", Key changes; "feat: Support dynamic
// batching for heterogeneous diffusion requests", AttentionMetadata).
//
// Design (one persistent CTA per SM, 6 warps):
//   warp 0      TMA producer: Q tile once per work item, then K/V tiles in
//               the order the MMAs consume them (K0, K1, V0, K2, V1, ...)
//               through a ring of shared-memory slots.
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma:
//               S = Q K^T (A, B from shared memory, fp32 into TMEM, double
//               buffered) and O += P V (P from TMEM as bf16, V from shared
//               memory, fp32 accumulator in TMEM).
//   warps 2..5  one thread per query row: read S from TMEM, online softmax
//               in fp32 (exp2 with the scale folded in), write P to TMEM,
//               rescale O in TMEM only when the row maximum grew by more
//               than 2^8, and finally normalise O and store bf16 rows.
// Work items (sequence, head, 128-row query tile) come from the
// length-ordered list of sched.cuh; every item is computed by one CTA in a
// fixed key-tile order, so results do not depend on the rest of the batch.
// Key columns past the sequence end are masked to -inf (P = 0 there); query
// rows past it are computed but never stored.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kTile = 128;          // query rows per item and keys per tile
constexpr int kThreads = 192;       // 6 warps
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;  // teardown after an abort (~0.2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units

template <int D>
struct Cfg {
  static constexpr int kHalfBytes = kTile * 64 * 2;         // 128 rows x 128 B
  static constexpr int kTileBytes = kTile * D * 2;          // one Q/K/V tile
  static constexpr int kSlots = D == 128 ? 5 : 10;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0, kQEmpty = 1, kSFull = 2, kSFree = 4, kPReady = 6,
                       kPVDone = 7, kFinal = 8, kSlotFull = 9, kSlotEmpty = 9 + kSlots;
  static constexpr int kNumBars = 9 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kSchedOff = (kMiscOff + 16 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kSchedOff + (2 * PA_MAX_BATCH + 1) * 4 + 1024;
  // TMEM columns
  static constexpr uint32_t kColS = 0;           // S buffers at 0 and 128
  static constexpr uint32_t kColO = 256;         // O: D columns
  static constexpr uint32_t kColP = 256 + D;     // P: 64 columns (128 bf16)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, kTile, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kTile, D, true);
  // V (MN-major): next 64-column half at LBO, next 8 keys at SBO = 1024.  With
  // D = 64 the MMA spans a single half and LBO is never used.
  static constexpr uint32_t kVLbo = D == 128 ? kHalfBytes : 1024;
};

struct TcParams {
  __nv_bfloat16 *out;
  const int32_t *cu_q, *cu_k;
  int batch, H, total_q, total_k, max_q, max_k;
  float scale_log2;
  int32_t *status;
};

struct ItemInfo {
  int q_row0;   // global row of the tile's first query
  int rows;     // valid query rows in the tile (1..128)
  int k0;       // global row of the sequence's first key
  int lk;       // keys of the sequence
  int nk;       // key tiles
  int head;
};

__device__ __forceinline__ ItemInfo item_info(const TcParams &p, const int32_t *order,
                                              const int32_t *prefix, int i) {
  const WorkItem w = sched_item(order, prefix, p.batch, p.H, i);
  int err;
  const SeqBounds sb = seq_bounds(p.cu_q, p.cu_k, w.seq, p.total_q, p.total_k, p.max_q,
                                  p.max_k, err);
  ItemInfo it;
  it.q_row0 = sb.q0 + w.tile * kTile;
  it.rows = min(kTile, sb.lq - w.tile * kTile);
  it.k0 = sb.k0;
  it.lk = sb.lk;
  it.nk = (sb.lk + kTile - 1) / kTile;
  it.head = w.head;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzle atoms)
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kQOff;
  const uint32_t sRing = base + C::kRingOff;
  auto bar = [&](int idx) -> uint32_t { return base + C::kBarOff + 8u * idx; };
  uint32_t *tmem_base_ptr = reinterpret_cast<uint32_t *>(gbase + C::kMiscOff);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(gbase + C::kMiscOff + 4);
  int32_t *order = reinterpret_cast<int32_t *>(gbase + C::kSchedOff);
  int32_t *prefix = order + PA_MAX_BATCH;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- set-up: barriers, TMEM, work list --------------------------------
  if (tid == 0) {
    mbar_init(bar(C::kQFull), 1);
    mbar_init(bar(C::kQEmpty), 1);
    mbar_init(bar(C::kSFull + 0), 1);
    mbar_init(bar(C::kSFull + 1), 1);
    mbar_init(bar(C::kSFree + 0), 128);
    mbar_init(bar(C::kSFree + 1), 128);
    mbar_init(bar(C::kPReady), 128);
    mbar_init(bar(C::kPVDone), 1);
    mbar_init(bar(C::kFinal), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kSlotFull + s), 1);
      mbar_init(bar(C::kSlotEmpty + s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(base + C::kMiscOff, C::kTmemCols);
  // the ring is free until the first load: use it for the build's temporaries
  int32_t *tmp = reinterpret_cast<int32_t *>(gbase + C::kRingOff);
  sched_build(order, prefix, tmp, tmp + PA_MAX_BATCH, p.cu_q, p.cu_k, p.batch, p.H, kTile,
              p.total_q, p.total_k, p.max_q, p.max_k, p.status, blockIdx.x == 0);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_base_ptr;
  const int n_items = prefix[p.batch];

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t q_loads = 0, slot_loads = 0;
      bool ok = true;
      auto load_kv = [&](const CUtensorMap *tm, int row, int head) -> bool {
        const uint32_t s = slot_loads % C::kSlots;
        const uint32_t use = slot_loads / C::kSlots;
        if (!bounded_wait(bar(C::kSlotEmpty + s), (use & 1u) ^ 1u, abort_flag, p.status,
                          kWaitLimit))
          return false;
        mbar_arrive_expect_tx(bar(C::kSlotFull + s), C::kTileBytes);
        const uint32_t dst = sRing + s * C::kTileBytes;
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(dst + hf * C::kHalfBytes, tm, bar(C::kSlotFull + s), hf * 64, head, row);
        ++slot_loads;
        return true;
      };
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const ItemInfo it = item_info(p, order, prefix, i);
        if (it.nk == 0) continue;
        if (!bounded_wait(bar(C::kQEmpty), (q_loads & 1u) ^ 1u, abort_flag, p.status,
                          kWaitLimit)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(C::kQFull), C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(sQ + hf * C::kHalfBytes, &tm_q, bar(C::kQFull), hf * 64, it.head,
                      it.q_row0);
        ++q_loads;
        for (int j = 0; j < it.nk && ok; ++j) {
          ok = load_kv(&tm_k, it.k0 + j * kTile, it.head);
          if (ok && j >= 1) ok = load_kv(&tm_v, it.k0 + (j - 1) * kTile, it.head);
        }
        if (ok) ok = load_kv(&tm_v, it.k0 + (it.nk - 1) * kTile, it.head);
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
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      uint32_t q_uses = 0, slot_uses = 0, g = 0;
      bool ok = true;
      // descriptors: Q/K K-major (SBO = 8 rows x 128 B), V MN-major
      // (LBO = next 64-column half, SBO = next 8 keys)
      auto issue_pv = [&](uint32_t gg, bool first) -> bool {
        if (!bounded_wait(bar(C::kPReady), gg & 1u, abort_flag, p.status, kWaitLimit))
          return false;
        const uint32_t s = slot_uses % C::kSlots;
        if (!bounded_wait(bar(C::kSlotFull + s), (slot_uses / C::kSlots) & 1u, abort_flag,
                          p.status, kWaitLimit))
          return false;
        fence_after_sync();
        const uint32_t v_addr = sRing + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(v_addr + kk * 16 * 128, C::kVLbo, 1024);
          mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8, bdesc, C::kIdescO,
                 (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(bar(C::kPVDone));
        mma_commit(bar(C::kSlotEmpty + s));
        ++slot_uses;
        return true;
      };
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const ItemInfo it = item_info(p, order, prefix, i);
        if (it.nk == 0) continue;
        if (!bounded_wait(bar(C::kQFull), q_uses & 1u, abort_flag, p.status, kWaitLimit)) {
          ok = false;
          break;
        }
        ++q_uses;
        for (int j = 0; j < it.nk && ok; ++j) {
          const uint32_t gg = g + j;
          const uint32_t buf = gg & 1u, use = gg >> 1;
          const uint32_t s = slot_uses % C::kSlots;
          ok = bounded_wait(bar(C::kSlotFull + s), (slot_uses / C::kSlots) & 1u, abort_flag,
                            p.status, kWaitLimit) &&
               bounded_wait(bar(C::kSFree + buf), (use & 1u) ^ 1u, abort_flag, p.status,
                            kWaitLimit);
          if (!ok) break;
          fence_after_sync();
          const uint32_t k_addr = sRing + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
            const uint64_t adesc = sdesc_sw128(sQ + off, 16, 1024);
            const uint64_t bdesc = sdesc_sw128(k_addr + off, 16, 1024);
            mma_ss(tmem + C::kColS + buf * kTile, adesc, bdesc, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kSFull + buf));
          mma_commit(bar(C::kSlotEmpty + s));
          ++slot_uses;
          if (j == it.nk - 1) mma_commit(bar(C::kQEmpty));
          if (j >= 1) ok = issue_pv(gg - 1, j == 1);
        }
        if (ok) ok = issue_pv(g + it.nk - 1, it.nk == 1);
        g += it.nk;
      }
      // every MMA issued so far has finished before TMEM is released
      if (g > 0 || q_uses > 0) {
        mma_commit(bar(C::kFinal));
        drain_wait(bar(C::kFinal), 0, kWaitLimit);
      }
    }
    __syncwarp();
  } else {
    // ================= softmax / correction / epilogue =================
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? sl2 : 1.f;
    uint32_t g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      const ItemInfo it = item_info(p, order, prefix, i);
      __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(it.q_row0 + row) * p.H + it.head) * D;
      const bool store = row < it.rows;
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
        const uint32_t gg = g + j;
        const uint32_t buf = gg & 1u, use = gg >> 1;
        ok = bounded_wait(bar(C::kSFull + buf), use & 1u, abort_flag, p.status, kWaitLimit);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        fence_after_sync();
        // all four 32-column loads in flight, then one wait
        uint32_t sr[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
          tmem_ld32(lane_base + C::kColS + buf * kTile + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_wait_ld();
        fence_before_sync();
        mbar_arrive(bar(C::kSFree + buf));
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
        if (j == it.nk - 1) {
          const int valid = it.lk - j * kTile;
#pragma unroll
          for (int c = 0; c < kTile / 2; ++c) {
            if (2 * c >= valid) x[c].x = -INFINITY;
            if (2 * c + 1 >= valid) x[c].y = -INFINITY;
          }
        }
        // row maximum: eight independent chains of 3-input max, fixed combine
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
          const float2 t = __ffma2_rn(x[c], mul2, negm2);
          const float2 pp = make_float2(ex2(t.x), ex2(t.y));
          sum8[c & 7] = __fadd2_rn(sum8[c & 7], pp);
          pk[c] = pack_bf16x2(pp.x, pp.y);
        }
        const float2 s01 = __fadd2_rn(__fadd2_rn(sum8[0], sum8[1]), __fadd2_rn(sum8[2], sum8[3]));
        const float2 s45 = __fadd2_rn(__fadd2_rn(sum8[4], sum8[5]), __fadd2_rn(sum8[6], sum8[7]));
        const float2 s8 = __fadd2_rn(s01, s45);
        const float sum = s8.x + s8.y;
        l = l * alpha + sum;
        if (j >= 1) {
          // PV of the previous tile must be done: it updates O and reads P
          ok = bounded_wait(bar(C::kPVDone), (gg - 1) & 1u, abort_flag, p.status, kWaitLimit);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          fence_after_sync();
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + C::kColO + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(lane_base + C::kColO + c * 32, r);
            }
          }
        }
        {
          uint32_t r[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = pk[e];
          tmem_st32(lane_base + C::kColP, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = pk[32 + e];
          tmem_st32(lane_base + C::kColP + 32, r);
        }
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::kPReady));
      }
      if (!ok) break;
      // epilogue: wait for the last PV, normalise, store the valid rows
      ok = bounded_wait(bar(C::kPVDone), (g + it.nk - 1) & 1u, abort_flag, p.status,
                        kWaitLimit);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::kColO + c * 32, r);
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
      g += it.nk;
    }
  }

  // ---- teardown -------------------------------------------------------------
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [rows, H, D] bf16 viewed as a 3-D tensor (D, H, rows); box 64 x 1 x 128
// with 128-byte swizzle: one 128-row, 64-column half tile per load.
bool make_map(CUtensorMap *map, const void *ptr, int rows, int H, int D) {
  EncodeTiledFn enc = encode_fn();
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

template <int D>
cudaError_t launch_tc(const VarlenArgs &a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.total_q, a.H, D) || !make_map(&mk, a.k, a.total_k, a.H, D) ||
      !make_map(&mv, a.v, a.total_k, a.H, D))
    return cudaErrorInvalidValue;
  TcParams p;
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
  const int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(varlen_attn_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  varlen_attn_tc_kernel<D><<<a.num_sms, kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_varlen_attn(const VarlenArgs &a, cudaStream_t stream) {
  return a.D == 64 ? launch_tc<64>(a, stream) : launch_tc<128>(a, stream);
}

}  // namespace pa
