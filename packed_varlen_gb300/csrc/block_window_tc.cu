// Block-window attention of the Token2Wav DiT on the 5th-generation tensor
// cores ("[Perf][Model] Use block-sparse attention in Qwen2.5-Omni Token2Wav
// DiT", Purpose and Change): frames are grouped in blocks; query i sees key j
// iff j < n and
//   -look_back <= block(j) - block(i) <= look_ahead.
//
// Work item: the query rows of one (batch entry, head) that fill one
// 128-lane tile, placed so that every 32-lane quadrant (the lanes one warp
// reads from TMEM) holds G rows: G = block * floor(32 / block) when a block
// fits in 32 rows (the DiT's 24-frame blocks: one block per quadrant, 8
// padding lanes), else G = 32.  A quadrant's rows then share one key window,
// so each softmax warp reads only that window's columns of S.  The item's
// rows together span one contiguous key range, fetched with TMA in chunks of
// at most N <= 256 keys; for the DiT every item is a single chunk: one
// S = Q K^T MMA (M = 128, N keys), one softmax per row and one O = P V MMA,
// with no rescaling.  Longer windows (long blocks, wide looks) loop over
// chunks with an online softmax whose running output is held in registers
// (the kMulti variant).
//
// A layer is small (n = 2400, H = 16, D = 64: 19.7 MB of q/k/v/out), so the
// kernel is built for memory-level parallelism and short per-item chains:
// one persistent CTA per SM keeps up to four items in flight in shared-memory
// slots, and the TMA producer issues every slot's loads as soon as the slot
// is free, so a whole layer's reads are in flight from the start; three
// softmax warpgroups work on three items at once (the DiT layer: 400 items of
// 4 blocks x 24 rows, at most three per CTA).
//
//   warp 0        TMA producer: per item Q once, then K and V chunk by chunk.
//   warp 1        allocates TMEM (512 columns) and issues the S = Q K^T MMAs
//                 in item order as each item's loads land.
//   warp 14       issues the O = P V MMAs in item order as each item's P is
//                 written, so a late load never holds up a ready PV.
//   warps 2-13    three softmax + epilogue groups of four warps, one thread
//                 per TMEM lane; group g takes the local items li = g mod 3.
//                 Each thread masks its row of S to the row's key interval
//                 (two integer compares per score, decided from n, block,
//                 look_back and look_ahead), writes P as bf16 over the first
//                 N/2 columns of S, and after the PV reads O, normalises and
//                 stores bf16.
// TMEM per slot: S at [0, N), P over [0, N/2), O at [o_off, o_off + D) with
// o_off >= N/2, so P and O live inside the columns S used and a slot costs
// max(N, o_off + D) columns (long windows at D = 128: O after S, where it
// accumulates over the chunks).  Keys outside [0, n) are zero-filled by TMA and
// never inside any row's interval.  Every wait is bounded.
//
// The kernel is launched with programmatic stream serialization: it starts
// while the previous kernel on the stream drains, sets up its barriers and
// TMEM and decodes its first item, and only the threads that touch global
// memory wait (griddepcontrol.wait) for that kernel's results: the producer
// before its first copy, the softmax warps before their first store.  The
// kernel's source is kept small (rolled loops over 32-column pieces, an
// out-of-line polling loop): it runs for a few microseconds, so instruction
// fetch on first use is part of its critical path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"
#include "tma_map.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kM = 128;                          // MMA rows (TMEM lanes)
constexpr int kMaxN = 256;                       // keys per chunk: MMA N and TMA box limit
constexpr int kMaxSlots = 4;
constexpr int kGroups = 3;                       // softmax warpgroups
constexpr int kThreads = (3 + 4 * kGroups) * 32; // producer, S issuer, softmax groups, PV issuer
constexpr int kPvWarp = 2 + 4 * kGroups;
constexpr int kTmemCols = 512;
constexpr int kBarsPerSlot = 9;
constexpr int kQFull = 0, kQEmpty = 1, kKFull = 2, kKvEmpty = 3, kSFull = 4, kPReady = 5,
              kOFull = 6, kTFree = 7, kVFull = 8;
constexpr int kBarBytes = (kMaxSlots * kBarsPerSlot + 2) * 8;
constexpr int kMiscBytes = 16;                   // TMEM base, abort flag
constexpr int kMaxSmem = 232448;
constexpr int kMinSmem = 120 * 1024;             // two CTAs never share an SM (TMEM)
constexpr long long kWaitLimit = 4000000000LL;   // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;   // teardown after an abort (~0.2 s)

struct BwTcParams {
  __nv_bfloat16 *out;
  int n, block, look_back, look_ahead, H, batch;
  int G;            // query rows per 32-lane quadrant (R = 4 G rows per item)
  int N;            // keys per chunk (multiple of 16, <= 256)
  int tiles;        // items per (batch entry, head): ceil(n / R)
  int n_items;
  int nslots, depth;
  int slot_bytes, k_off, v_off;   // shared memory of a slot
  int slot_cols, o_off;           // TMEM of a slot
  int bar_off;
  uint32_t idesc_s, idesc_o;
  float scale_log2;
  int32_t *status;
};

struct BwItem {
  int bi, h, r0, rows;   // rows [r0, r0 + rows) of the entry, rows <= 4 G
  int kb, nc;            // first key of the window, chunks
};

__device__ __forceinline__ BwItem bw_item(const BwTcParams &p, int item) {
  BwItem it;
  it.h = item % p.H;
  const int rest = item / p.H;
  const int t = rest % p.tiles;
  it.bi = rest / p.tiles;
  it.r0 = t * 4 * p.G;
  it.rows = min(4 * p.G, p.n - it.r0);
  const int fb = it.r0 / p.block, lb = (it.r0 + it.rows - 1) / p.block;
  long long kb = (static_cast<long long>(fb) - p.look_back) * p.block;
  long long ke = (static_cast<long long>(lb) + 1 + p.look_ahead) * p.block;
  if (kb < 0) kb = 0;
  if (ke > p.n) ke = p.n;
  it.kb = static_cast<int>(kb);
  it.nc = (static_cast<int>(ke) - it.kb + p.N - 1) / p.N;   // 32-bit: ke <= n
  return it;
}

// Per-slot counters kept in registers (nslots <= 4).
__device__ __forceinline__ uint32_t cnt_get(const uint32_t (&c)[kMaxSlots], int s) {
  return s == 0 ? c[0] : s == 1 ? c[1] : s == 2 ? c[2] : c[3];
}
__device__ __forceinline__ void cnt_add(uint32_t (&c)[kMaxSlots], int s, uint32_t v) {
#pragma unroll
  for (int i = 0; i < kMaxSlots; ++i) c[i] += (i == s) ? v : 0u;
}

constexpr int kFastCols = 32;   // widest window of the one-window fast path

// Bounded mbarrier wait: the first poll inline, the polling loop out of
// line (it only runs while the warp has nothing else to do), which keeps the
// many wait sites of this short kernel from inflating its code.
__device__ __noinline__ bool bw_wait_slow(uint32_t bar, uint32_t parity,
                                          volatile int32_t *abort_flag, int32_t *status) {
  return bounded_wait(bar, parity, abort_flag, status, kWaitLimit);
}
__device__ __forceinline__ bool bw_wait(uint32_t bar, uint32_t parity,
                                        volatile int32_t *abort_flag, int32_t *status) {
  return mbar_try_wait(bar, parity) || bw_wait_slow(bar, parity, abort_flag, status);
}

// Softmax pieces of 32 S columns (keys col0 .. col0 + 31 of the chunk).
// Maximum of the scaled scores inside the row's columns [a, e).
__device__ __forceinline__ float max32(const uint32_t (&r)[32], int col0, int a, int e,
                                       bool pos_scale, float sl2, float mx) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float x = __uint_as_float(r[j]);
    if (!pos_scale) x *= sl2;
    mx = fmaxf(mx, (col0 + j >= a && col0 + j < e) ? x : -INFINITY);
  }
  return mx;
}
// P = exp2(scaled score * mul + negm) inside [a, e), 0 elsewhere, stored as 16
// bf16 pairs at TMEM address `taddr`; returns the sum of the 32 values.
__device__ __forceinline__ float put_p32(const uint32_t (&r)[32], int col0, int a, int e,
                                         bool pos_scale, float sl2, float mul, float negm,
                                         uint32_t taddr) {
  uint32_t pk[16];
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
    if (!pos_scale) {
      x0 *= sl2;
      x1 *= sl2;
    }
    const int c0 = col0 + 2 * j;
    const float p0 = (c0 >= a && c0 < e) ? ex2(fmaf(x0, mul, negm)) : 0.f;
    const float p1 = (c0 + 1 >= a && c0 + 1 < e) ? ex2(fmaf(x1, mul, negm)) : 0.f;
    sum += p0 + p1;
    pk[j] = pack_bf16x2(p0, p1);
  }
  tmem_st16(taddr, pk);
  return sum;
}

// kMulti: some item window is longer than one chunk (online softmax over
// chunks, running output in registers); otherwise every item is one chunk.
template <int D, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
    block_window_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const BwTcParams p) {
  // long windows at D = 128: the running output of the chunks stays in TMEM
  // (after S in the slot), accumulated by the PV MMAs; 128 fp32 registers
  // per thread would spill
  constexpr bool kOInTmem = kMulti && D == 128;
  // D = 128 reads O for the epilogue 32 columns at a time (all 128 at once
  // would spill); D = 64 reads its 64 columns in one go
  constexpr bool kOPieces = D == 128;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) {   // descriptor fetches overlap the set-up below
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {   // 128-byte swizzle atoms need a 1024-byte aligned base
    if (threadIdx.x == 0) record_error(p.status, PA_DEVICE_ERR_SMEM_ALIGN);
    return;
  }
  auto bar = [&](int s, int role) -> uint32_t {
    return base + p.bar_off + 8u * (s * kBarsPerSlot + role);
  };
  const uint32_t final_bar = base + p.bar_off + 8u * (kMaxSlots * kBarsPerSlot);
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem_raw + p.bar_off + kBarBytes);
  volatile int32_t *abort_flag =
      reinterpret_cast<volatile int32_t *>(smem_raw + p.bar_off + kBarBytes + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = p.nslots;
  const int N = p.N;
  const int G = p.G;

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(bar(s, kQFull), 1);
      mbar_init(bar(s, kQEmpty), 1);
      mbar_init(bar(s, kKFull), 1);
      mbar_init(bar(s, kVFull), 1);
      mbar_init(bar(s, kKvEmpty), 1);
      mbar_init(bar(s, kSFull), 1);
      mbar_init(bar(s, kPReady), 128);
      mbar_init(bar(s, kOFull), 1);
      mbar_init(bar(s, kTFree), 128);
    }
    mbar_init(final_bar, 1);
    mbar_init(final_bar + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_ptr), kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_ptr;
  // the next kernel on the stream may start its own set-up now; this
  // kernel's global reads and writes wait (griddep_wait) for the previous
  // kernel, so inputs it wrote are visible and outputs it may still read are
  // not overwritten before it finishes
  griddep_launch_dependents();

  auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
    const bool w = bw_wait(b, parity, abort_flag, p.status);
    return __all_sync(0xffffffffu, w);
  };
  // local items of this CTA: li = 0, 1, ...; item = blockIdx.x + li * gridDim.x
  const int n_local =
      p.n_items > static_cast<int>(blockIdx.x)
          ? (p.n_items - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
          : 0;

  if (warp == 0) {
    // ================= TMA producer =================
    const bool lead = elect_one();
    uint32_t kvc[kMaxSlots] = {0, 0, 0, 0};   // K copies per slot
    uint32_t vc[kMaxSlots] = {0, 0, 0, 0};    // V copies per slot
    int q_loads = 0;
    bool ok = true;
    const uint32_t q_bytes = (G == 32 ? kM : 4u * G) * D * 2u;
    const uint32_t kv_bytes = static_cast<uint32_t>(N) * D * 2u;   // K or V of one chunk
    // Q of local item li, after the slot's previous item has released it
    auto load_q = [&](int li, const BwItem &it) -> bool {
      const int s = li % ns;
      const uint32_t slot = base + s * p.slot_bytes;
      if (!wait_all(bar(s, kQEmpty), ((li / ns) & 1) ^ 1)) return false;
      if (li == 0) griddep_wait();
      if (lead) {
        mbar_arrive_expect_tx(bar(s, kQFull), q_bytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          if (G == 32) {
            tma_load_4d(slot + hf * (kM * 128), &tm_q, bar(s, kQFull), hf * 64, it.h, it.r0,
                        it.bi);
          } else {
            // quadrant q's G rows at lanes [32 q, 32 q + G)
            for (int q = 0; q < 4; ++q)
              tma_load_4d(slot + hf * (kM * 128) + q * (32 * 128), &tm_q, bar(s, kQFull),
                          hf * 64, it.h, it.r0 + q * G, it.bi);
          }
        }
      }
      ++q_loads;
      return true;
    };
    // K of chunk c, after the slot's previous chunk has released its K/V
    auto load_k = [&](int s, const BwItem &it, int c) -> bool {
      if (!wait_all(bar(s, kKvEmpty), (cnt_get(kvc, s) & 1u) ^ 1u)) return false;
      if (lead) {
        mbar_arrive_expect_tx(bar(s, kKFull), kv_bytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_4d(base + s * p.slot_bytes + p.k_off + hf * (N * 128), &tm_k, bar(s, kKFull),
                      hf * 64, it.h, it.kb + c * N, it.bi);
      }
      cnt_add(kvc, s, 1u);
      return true;
    };
    // V of chunk c (its slot was waited for by load_k)
    auto load_v = [&](int s, const BwItem &it, int c) {
      if (lead) {
        mbar_arrive_expect_tx(bar(s, kVFull), kv_bytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_4d(base + s * p.slot_bytes + p.v_off + hf * (N * 128), &tm_v, bar(s, kVFull),
                      hf * 64, it.h, it.kb + c * N, it.bi);
      }
      cnt_add(vc, s, 1u);
    };
    if constexpr (!kMulti) {
      // One chunk per item.  Items go in windows of ns (one per slot); a
      // window's Q and K copies are issued before its V copies.  The loads
      // are DRAM-bound and land roughly in issue order, so the scores and
      // softmax of every item of the window run while the V rows stream in,
      // and only the PV and the epilogue follow the last bytes.
      for (int w0 = 0; w0 < n_local && ok; w0 += ns) {
        const int w1 = min(n_local, w0 + ns);
        for (int li = w0; li < w1 && ok; ++li) {
          const BwItem it = bw_item(p, blockIdx.x + li * gridDim.x);
          ok = load_q(li, it) && load_k(li % ns, it, 0);
        }
        for (int li = w0; li < w1 && ok; ++li)
          load_v(li % ns, bw_item(p, blockIdx.x + li * gridDim.x), 0);
      }
    } else {
      for (int li = 0; li < n_local && ok; ++li) {
        const BwItem it = bw_item(p, blockIdx.x + li * gridDim.x);
        ok = load_q(li, it);
        for (int c = 0; c < it.nc && ok; ++c) {
          ok = load_k(li % ns, it, c);
          if (ok) load_v(li % ns, it, c);
        }
      }
    }
    if (!ok) {
      // give the copies already issued a bounded chance to land
      for (int s = 0; s < ns; ++s) {
        const uint32_t u = cnt_get(kvc, s), uv = cnt_get(vc, s);
        if (u) drain_wait(bar(s, kKFull), (u - 1) & 1u, kDrainLimit);
        if (uv) drain_wait(bar(s, kVFull), (uv - 1) & 1u, kDrainLimit);
        const int qn = (q_loads + ns - 1 - s) / ns;   // Q loads into slot s
        if (qn) drain_wait(bar(s, kQFull), (qn - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp == 1 || warp == kPvWarp) {
    // ================= MMA issuers: S (warp 1), PV (last warp) =================
    const bool lead = elect_one();
    bool ok = true, issued = false;
    auto issue_s = [&](int s, uint32_t d_s) {
      const uint32_t slot = base + s * p.slot_bytes;
      const uint64_t qdesc = sdesc_sw128(slot, 16, 1024);
      const uint64_t kdesc = sdesc_sw128(slot + p.k_off, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oq = ((kk >> 2) * (kM * 128) + (kk & 3) * 32) >> 4;
        const uint32_t okk = ((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4;
        if (lead) mma_ss(d_s, qdesc + oq, kdesc + okk, p.idesc_s, kk > 0 ? 1u : 0u);
      }
      issued = true;
    };
    // acc: the first MMA adds to O (a running output in TMEM) instead of
    // overwriting it
    auto issue_pv = [&](int s, uint32_t d_s, bool acc) {
      const uint32_t slot = base + s * p.slot_bytes;
      const uint64_t vdesc = sdesc_sw128(slot + p.v_off, D == 128 ? N * 128 : 1024, 1024);
      for (int kk = 0; kk < N / 16; ++kk) {
        if (lead)
          mma_ts(d_s + p.o_off, d_s + kk * 8, vdesc + ((kk * 16 * 128) >> 4), p.idesc_o,
                 (kk > 0 || acc) ? 1u : 0u);
      }
    };
    if constexpr (!kMulti) {
      if (warp == 1) {
        for (int li = 0; li < n_local && ok; ++li) {
          const int s = li % ns;
          const uint32_t ph = (li / ns) & 1;
          if (!wait_all(bar(s, kQFull), ph) || !wait_all(bar(s, kTFree), ph ^ 1u) ||
              !wait_all(bar(s, kKFull), ph)) {
            ok = false;
            break;
          }
          fence_after_sync();
          issue_s(s, tmem + s * p.slot_cols);
          if (lead) {
            mma_commit(bar(s, kSFull));
            mma_commit(bar(s, kQEmpty));
          }
        }
      } else {
        for (int li = 0; li < n_local && ok; ++li) {
          const int s = li % ns;
          if (!wait_all(bar(s, kPReady), (li / ns) & 1) || !wait_all(bar(s, kVFull), (li / ns) & 1)) {
            ok = false;
            break;
          }
          fence_after_sync();
          issue_pv(s, tmem + s * p.slot_cols, false);
          issued = true;
          if (lead) {
            mma_commit(bar(s, kOFull));
            mma_commit(bar(s, kKvEmpty));
          }
        }
      }
    } else if (warp == 1) {
      // chunks in order, one at a time; per-slot chunk counters
      uint32_t kvc[kMaxSlots] = {0, 0, 0, 0};
      for (int li = 0; li < n_local && ok; ++li) {
        const int s = li % ns;
        const BwItem it = bw_item(p, blockIdx.x + li * gridDim.x);
        if (!wait_all(bar(s, kQFull), (li / ns) & 1)) {
          ok = false;
          break;
        }
        const uint32_t d_s = tmem + s * p.slot_cols;
        for (int c = 0; c < it.nc; ++c) {
          const uint32_t u = cnt_get(kvc, s);
          if (!wait_all(bar(s, kTFree), (u & 1u) ^ 1u) || !wait_all(bar(s, kKFull), u & 1u)) {
            ok = false;
            break;
          }
          fence_after_sync();
          issue_s(s, d_s);
          if (lead) {
            mma_commit(bar(s, kSFull));
            if (c == it.nc - 1) mma_commit(bar(s, kQEmpty));
          }
          if (!wait_all(bar(s, kPReady), u & 1u) || !wait_all(bar(s, kVFull), u & 1u)) {
            ok = false;
            break;
          }
          fence_after_sync();
          issue_pv(s, d_s, kOInTmem && c > 0);
          if (lead) {
            mma_commit(bar(s, kOFull));
            mma_commit(bar(s, kKvEmpty));
          }
          cnt_add(kvc, s, 1u);
        }
      }
    }
    // every MMA issued has finished before TMEM is released
    if (issued) {
      const uint32_t fb = final_bar + (warp == 1 ? 0u : 8u);
      if (lead) mma_commit(fb);
      drain_wait(fb, 0, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ================= softmax + epilogue =================
    const int g = (warp - 2) >> 2;
    const int quad = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? sl2 : 1.f;
    uint32_t kvc[kMaxSlots] = {0, 0, 0, 0};   // kMulti: per-slot chunk counters
    bool ok = true, waited = false;
    for (int li = 0; li < n_local && ok; ++li) {
      const int s = li % ns;
      const BwItem it = bw_item(p, blockIdx.x + li * gridDim.x);
      if (li % kGroups != g) {
        if constexpr (kMulti) cnt_add(kvc, s, static_cast<uint32_t>(it.nc));
        continue;
      }
      // this thread's query row: lane `lane` of quadrant `quad`
      const int rq = quad * G + lane;                 // row within the item
      const bool valid = lane < G && rq < it.rows;
      const int i = it.r0 + rq;
      long long lo = 0, hi = 0;   // the row's key interval [lo, hi)
      if (valid) {
        const long long b = i / p.block;
        lo = (b - p.look_back) * static_cast<long long>(p.block);
        hi = (b + 1 + p.look_ahead) * static_cast<long long>(p.block);
        if (lo < 0) lo = 0;
        if (hi > p.n) hi = p.n;
      }
      const uint32_t col_s = s * p.slot_cols, col_o = col_s + p.o_off;
      __nv_bfloat16 *dst =
          p.out + ((static_cast<int64_t>(it.bi) * p.n + (valid ? i : 0)) * p.H + it.h) * D;
      float m_run = -INFINITY, l_run = 0.f;
      float acc[kMulti && !kOInTmem ? D : 1];
      for (int c = 0; c < it.nc; ++c) {
        const uint32_t u = kMulti ? cnt_get(kvc, s) : static_cast<uint32_t>(li / ns);
        // this row's columns [a, e) of the chunk, the warp's union in 32-column
        // pieces [w0, w1) (a piece past N reads columns inside the slot and
        // masks them) and the fast-path test below depend only on the block
        // arithmetic: they are settled before the scores are waited for
        const long long kc = static_cast<long long>(it.kb) + static_cast<long long>(c) * N;
        int a = static_cast<int>(max(0LL, min(static_cast<long long>(N), lo - kc)));
        int e = static_cast<int>(max(0LL, min(static_cast<long long>(N), hi - kc)));
        if (a >= e) {
          a = N;
          e = 0;
        }
        const int w0 = __reduce_min_sync(0xffffffffu, a) >> 5;
        const int w1 = (__reduce_max_sync(0xffffffffu, e) + 31) >> 5;
        // Fast path: every row of the warp that has keys in this chunk has the
        // same interval [ua, ue), starting on an 8-column boundary and at most
        // kFastCols wide (the DiT's own-block layers: one 24-frame block per
        // quadrant).  The warp then reads exactly those columns once, keeps
        // them in registers for both passes, and masks only a ragged last
        // 8-column group; rows without keys (padding lanes) compute values
        // that are never stored.
        const int ua = __reduce_max_sync(0xffffffffu, a < e ? a : -1);
        const int ub = __reduce_min_sync(0xffffffffu, a < e ? a : 0x7fffffff);
        const int ue = __reduce_max_sync(0xffffffffu, a < e ? e : -1);
        const int uf = __reduce_min_sync(0xffffffffu, a < e ? e : 0x7fffffff);
        const bool fast = !kMulti && pos_scale && ua >= 0 && ua == ub && ue == uf &&
                          (ua & 7) == 0 && ue - ua <= kFastCols;
        if (!wait_all(bar(s, kSFull), u & 1u)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const int ng = fast ? (ue - ua + 7) >> 3 : 0;   // 8-column groups
        uint32_t rw[kFastCols];
        float mx = -INFINITY;
        if (fast) {
#pragma unroll
          for (int g8 = 0; g8 < kFastCols / 8; ++g8)
            if (g8 < ng) tmem_ld8(lane_base + col_s + ua + g8 * 8, &rw[8 * g8]);
          tmem_wait_ld();
          if ((ue - ua) & 7) {   // keys past the interval in the last group
#pragma unroll
            for (int j = 0; j < kFastCols; ++j)
              if (j >= ue - ua) rw[j] = __float_as_uint(-INFINITY);
          }
          float mg[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int g8 = 0; g8 < kFastCols / 8; ++g8) {
            if (g8 < ng) {
              const uint32_t *v = &rw[8 * g8];
              const float m3 = fmax3(fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]),
                                           __uint_as_float(v[2])),
                                     fmax3(__uint_as_float(v[3]), __uint_as_float(v[4]),
                                           __uint_as_float(v[5])),
                                     fmaxf(__uint_as_float(v[6]), __uint_as_float(v[7])));
              mg[g8 & 1] = fmaxf(mg[g8 & 1], m3);
            }
          }
          mx = fmaxf(mg[0], mg[1]) * sl2;
        } else {
#pragma unroll 1
          for (int pc = w0; pc < w1; ++pc) {
            uint32_t r[32];
            tmem_ld32(lane_base + col_s + pc * 32, r);
            tmem_wait_ld();
            mx = max32(r, pc * 32, a, e, pos_scale, sl2, mx);
          }
        }
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2((m_run - m_use) * mul);   // 0 while nothing was seen
        const float negm = -m_use * mul;
        if constexpr (kOInTmem) {
          // the running O (chunks before c; their PVs are done, waited for
          // below) brought to the new maximum before this chunk's PV adds to it
          if (c > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t r[32];
              tmem_ld32(lane_base + col_o + cc * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              tmem_st32(lane_base + col_o + cc * 32, r);
            }
          }
        }
        // P of keys [32 i, 32 i + 32) goes to P columns [16 i, 16 i + 16),
        // which hold S columns of pieces <= i, read before the store; outside
        // the union P is 0 (stored after every read of the union, since those
        // columns may overlap its S columns)
        float lsum = 0.f;
        if (fast) {
          // P of the interval's keys over P columns [ua / 2, ua / 2 + 4 ng),
          // 0 over the rest of [0, N / 2) (after the interval was read)
          const float2 sl22 = make_float2(sl2, sl2), negm2 = make_float2(negm, negm);
          float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int g8 = 0; g8 < kFastCols / 8; ++g8) {
            if (g8 < ng) {
              uint32_t pk[4];
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const float2 tt = __ffma2_rn(
                    make_float2(__uint_as_float(rw[8 * g8 + 2 * jj]),
                                __uint_as_float(rw[8 * g8 + 2 * jj + 1])),
                    sl22, negm2);
                const float2 pp = make_float2(ex2(tt.x), ex2(tt.y));
                s2 = __fadd2_rn(s2, pp);
                pk[jj] = pack_bf16x2(pp.x, pp.y);
              }
              tmem_st4(lane_base + col_s + (ua >> 1) + 4 * g8, pk);
            }
          }
          lsum = s2.x + s2.y;
          // zeros over [0, p0) and [p1, N / 2) with the widest stores that
          // sit on a multiple of their own width (every bound is a multiple
          // of 4; a TMEM store costs about the same whatever its width)
          const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          const int p0 = ua >> 1, p1 = (ua >> 1) + 4 * ng;
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {
            int x = part == 0 ? 0 : p1;
            const int x1 = part == 0 ? p0 : N / 2;
#pragma unroll 1
            while (x < x1) {
              if ((x & 15) == 0 && x + 16 <= x1) {
                tmem_st16(lane_base + col_s + x, z);
                x += 16;
              } else if ((x & 7) == 0 && x + 8 <= x1) {
                tmem_st8(lane_base + col_s + x, z);
                x += 8;
              } else {
                tmem_st4(lane_base + col_s + x, z);
                x += 4;
              }
            }
          }
        } else {
#pragma unroll 1
          for (int pc = w0; pc < w1; ++pc) {
            uint32_t r[32];
            tmem_ld32(lane_base + col_s + pc * 32, r);
            tmem_wait_ld();
            lsum += put_p32(r, pc * 32, a, e, pos_scale, sl2, mul, negm,
                            lane_base + col_s + pc * 16);
          }
          const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
          for (int pc = 0; pc < (N + 31) / 32; ++pc)
            if (pc < w0 || pc >= w1) tmem_st16(lane_base + col_s + pc * 16, z);
        }
        l_run = l_run * alpha + lsum;
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(s, kPReady));
        // O of this chunk
        if (!wait_all(bar(s, kOFull), u & 1u)) {
          ok = false;
          break;
        }
        fence_after_sync();
        if constexpr (kOPieces) {
          // O / l of the last chunk, 32 columns at a time
          if (c == it.nc - 1) {
            if (!waited) {
              griddep_wait();
              waited = true;
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t r[32];
              tmem_ld32(lane_base + col_o + cc * 32, r);
              tmem_wait_ld();
              if (valid) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  uint4 w;
                  w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv,
                                    __uint_as_float(r[8 * v + 1]) * inv);
                  w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv,
                                    __uint_as_float(r[8 * v + 3]) * inv);
                  w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv,
                                    __uint_as_float(r[8 * v + 5]) * inv);
                  w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv,
                                    __uint_as_float(r[8 * v + 7]) * inv);
                  d4[v] = w;
                }
              }
            }
          }
          fence_before_sync();
          mbar_arrive(bar(s, kTFree));   // S and P may take the next chunk or item
          m_run = m_new;
          cnt_add(kvc, s, 1u);
          continue;
        }
        uint32_t o[D / 32][32];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_base + col_o + cc * 32, o[cc]);
        tmem_wait_ld();
        fence_before_sync();
        mbar_arrive(bar(s, kTFree));   // the slot's TMEM may take the next chunk or item
        if (!waited) {
          griddep_wait();
          waited = true;
        }
        if (!kMulti || it.nc == 1) {
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          if (valid) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(o[cc][8 * v + 0]) * inv,
                                  __uint_as_float(o[cc][8 * v + 1]) * inv);
                w.y = pack_bf16x2(__uint_as_float(o[cc][8 * v + 2]) * inv,
                                  __uint_as_float(o[cc][8 * v + 3]) * inv);
                w.z = pack_bf16x2(__uint_as_float(o[cc][8 * v + 4]) * inv,
                                  __uint_as_float(o[cc][8 * v + 5]) * inv);
                w.w = pack_bf16x2(__uint_as_float(o[cc][8 * v + 6]) * inv,
                                  __uint_as_float(o[cc][8 * v + 7]) * inv);
                d4[v] = w;
              }
            }
          }
        } else if constexpr (kMulti && !kOInTmem) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[cc * 32 + j] =
                  (c == 0 ? 0.f : acc[cc * 32 + j] * alpha) + __uint_as_float(o[cc][j]);
        }
        m_run = m_new;
        if constexpr (kMulti) cnt_add(kvc, s, 1u);
      }
      if (!ok) break;
      if constexpr (kMulti && !kOInTmem) {
        if (it.nc > 1 && valid) {
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) {
            uint4 w;
            w.x = pack_bf16x2(acc[8 * v + 0] * inv, acc[8 * v + 1] * inv);
            w.y = pack_bf16x2(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv);
            w.z = pack_bf16x2(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv);
            w.w = pack_bf16x2(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv);
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
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// [batch, n, H, D] bf16 viewed as a 4-D tensor (D, H, n, batch); box
// 64 x 1 x rows x 1 with 128-byte swizzle: one 64-column half of `rows`
// tokens of one head.  Rows outside [0, n) of an entry read as zero.
bool make_map_4d(CUtensorMap *map, const void *ptr, int batch, int n, int H, int D, int rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(n) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Tiling of one launch: G rows per quadrant (R = 4 G per item), keys per
// chunk N and the slot layout.  Returns whether any item window needs more
// than one chunk.
bool plan(const BlockWindowArgs &a, BwTcParams &p) {
  const int D = a.D;
  p.G = a.block <= 32 ? a.block * (32 / a.block) : 32;
  const int R = 4 * p.G;
  // blocks a tile of R rows touches: R / block when each quadrant holds whole
  // blocks, else up to ceil((R - 1) / block) + 1
  const long long span = a.block <= 32 ? R / a.block : (R - 1 + a.block - 1) / a.block + 1;
  long long W = (span + a.look_back + a.look_ahead) * static_cast<long long>(a.block);
  if (W > a.n) W = a.n;
  p.N = W >= kMaxN ? kMaxN : round_up(static_cast<int>(W), 16);
  const bool multi = W > p.N;
  if (multi && D == 128) {
    // the running output stays in TMEM across chunks: after S, not inside it
    p.o_off = round_up(p.N, 32);
    p.slot_cols = p.o_off + D;
  } else {
    p.o_off = round_up(p.N / 2, 32);
    p.slot_cols = round_up(p.N > p.o_off + D ? p.N : p.o_off + D, 32);
  }
  const int q_bytes = kM * D * 2, kv = p.N * D * 2;
  p.slot_bytes = q_bytes + 2 * kv;
  p.k_off = q_bytes;
  p.v_off = q_bytes + kv;
  int slots = kTmemCols / p.slot_cols;
  const int by_smem = (kMaxSmem - kBarBytes - kMiscBytes) / p.slot_bytes;
  if (slots > by_smem) slots = by_smem;
  if (slots > kMaxSlots) slots = kMaxSlots;
  p.nslots = slots;
  p.depth = slots < kGroups ? slots : kGroups;
  p.tiles = static_cast<int>((static_cast<long long>(a.n) + R - 1) / R);
  p.n_items = static_cast<int>(static_cast<long long>(p.tiles) * a.H * a.batch);
  p.bar_off = p.nslots * p.slot_bytes;
  p.idesc_s = idesc_bf16_f32(kM, p.N, false);
  p.idesc_o = idesc_bf16_f32(kM, D, true);
  return multi;
}

template <int D, bool kMulti>
cudaError_t launch_tc(const BlockWindowArgs &a, const BwTcParams &p, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map_4d(&mq, a.q, a.batch, a.n, a.H, D, p.G == 32 ? kM : p.G) ||
      !make_map_4d(&mk, a.k, a.batch, a.n, a.H, D, p.N) ||
      !make_map_4d(&mv, a.v, a.batch, a.n, a.H, D, p.N))
    return cudaErrorInvalidValue;
  int smem = p.bar_off + kBarBytes + kMiscBytes;
  if (smem < kMinSmem) smem = kMinSmem;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(
      reinterpret_cast<const void *>(block_window_tc_kernel<D, kMulti>), kMaxSmem, configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items < a.num_sms ? p.n_items : a.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, block_window_tc_kernel<D, kMulti>, mq, mk, mv, p);
}

}  // namespace

cudaError_t launch_block_window_attn(const BlockWindowArgs &a, cudaStream_t stream) {
  BwTcParams p{};
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.n = a.n;
  p.block = a.block;
  p.look_back = a.look_back;
  p.look_ahead = a.look_ahead;
  p.H = a.H;
  p.batch = a.batch;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  const bool multi = plan(a, p);
  if (static_cast<long long>(p.tiles) * a.H * a.batch > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.D == 64)
    return multi ? launch_tc<64, true>(a, p, stream) : launch_tc<64, false>(a, p, stream);
  return multi ? launch_tc<128, true>(a, p, stream) : launch_tc<128, false>(a, p, stream);
}

}  // namespace pa
