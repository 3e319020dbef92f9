// Batch-invariant packed-M linear layer on the 5th-generation tensor cores:
//
//   y[m, n] = sum_k x[m, k] * w[n, k]  (+ bias[n])
//
// with bf16 x, w, bias and y and fp32 accumulation.  The packed path runs
// the projections of every request at once on the flat [total_tokens, C]
// activations, and its batched and serial outputs are bit-identical because
// these GEMMs give a row the same result whatever the packed M is ("feat:
// Support dynamic batching for heterogeneous diffusion requests", packed
// varlen step batching: Setup, Determinism, and Notes, item 1).
//
// Batch invariance by construction: one tile shape (256 x 256 x 64 per CTA
// pair) for every M, no split-K, K walked in the same order in every tile, and an epilogue
// that treats each row alone.  A row's result therefore depends only on its
// own x row, w and bias: packed or alone, at any row offset, the bits agree.
//
// Kernel: persistent, one CTA per SM, CTAs in clusters of two that work as a
// cta_group::2 pair on 256 x 256 output tiles, six warps each.  One MMA
// (M = 256, N = 256, K = 16) spans the pair: each CTA holds 128 rows of the
// x tile and one 128-row half of the w tile in its own shared memory, loaded
// by its own TMA from this GPU's memory (no CTA writes another's shared
// memory), and receives its 128 output rows in its own TMEM.  Per CTA that is the L2
// traffic of a 128 x 256 tile with only half of w, and one MMA instruction
// per pair instead of two.
//   warp 0      TMA producer (both CTAs) into a kStages-deep ring; both
//               CTAs count their bytes on the even CTA's full barrier.
//   warp 1      allocates TMEM in both CTAs (a collective pair allocation);
//               in the even CTA it issues the MMAs into one of two TMEM
//               accumulators (2 x 256 fp32 columns) and frees each ring slot
//               in both CTAs with one commit per CTA.
//   warps 2-5   drain a finished accumulator (each warp its TMEM lane
//               quadrant), add the bias, round to bf16 and store, while the
//               MMA warp fills the other; each warp then reports the
//               accumulator free on the even CTA's barrier.
// Warps 0 and 1 run their loops warp-wide and one elected lane issues each
// copy, MMA and commit, so MMA operands are warp-uniform.  Tile pairs go
// round-robin over the clusters, N-block fastest, so a wave shares x rows and
// w stays in L2.  Every wait is bounded; a timeout records
// PA_DEVICE_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"
#include "tma_map.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 64;   // kBM rows per CTA, kBN columns per pair
constexpr int kStages = 6;
constexpr int kCluster = 2;                     // the CTA pair of one MMA
constexpr int kThreads = 192;                   // TMA, MMA, 4 epilogue warps
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;  // teardown after an abort (~0.2 s)

struct GemmCfg {
  static constexpr int kABytes = kBM * kBK * 2;                // 16 KB: 128 x rows x 128 B
  static constexpr int kBBytes = (kBN / kCluster) * kBK * 2;   // 16 KB: 128 w rows x 128 B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kFull = 0, kEmpty = kStages, kAccFull = 2 * kStages,
                       kAccEmpty = 2 * kStages + 2, kFinal = 2 * kStages + 4;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16;
  static constexpr uint32_t kTmemCols = 2 * kBN;
  // A (x) and B (w) both K-major; M spans the pair
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kCluster * kBM, kBN, false);
};
static_assert(GemmCfg::kSmemBytes <= 232448, "shared memory plan exceeds the per-CTA limit");

struct GemmParams {
  const __nv_bfloat16 *bias;  // [N] or nullptr
  __nv_bfloat16 *y;           // [M, N]
  int M, N, K;
  int tiles_n, n_pairs, k_blocks;   // n_pairs: (pair of 128-row blocks, N block)
  int32_t *status;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// bounded_wait with cluster-scope acquire, for barriers the other CTA of the
// pair (or its TMA and MMA completions) arrives on.
__device__ __forceinline__ bool bounded_wait_cl(uint32_t bar, uint32_t parity,
                                                volatile int32_t *abort_flag, int32_t *status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimit) {
      *abort_flag = 1;
      record_error(status, PA_DEVICE_ERR_TIMEOUT);
      return false;
    }
  }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    linear_bf16_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w, const GemmParams p) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need a 1024-byte aligned base.  Both CTAs of a
  // pair run the same code on the same layout, so both skip or neither.
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) record_error(p.status, PA_DEVICE_ERR_SMEM_ALIGN);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * i; };
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem_raw + C::kMiscOff);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem_raw + C::kMiscOff + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(C::kFull + s), 1);    // the leader's expect_tx; bytes of both CTAs
      mbar_init(bar(C::kEmpty + s), 1);   // one commit from the leader's MMA warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kAccFull + b), 1);
      mbar_init(bar(C::kAccEmpty + b), 4 * kCluster);   // every epilogue warp of the pair
    }
    mbar_init(bar(C::kFinal), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(base + C::kMiscOff, C::kTmemCols);
  fence_before_sync();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();   // barriers of both CTAs initialised before any remote use
  fence_after_sync();
  const uint32_t tmem = *tmem_ptr;
  const int cl = blockIdx.x / kCluster, n_cl = gridDim.x / kCluster;

  if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
    const bool lead = elect_one();
    if (lead) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
    }
    uint32_t loads = 0;
    bool ok = true;
    for (int tp = cl; tp < p.n_pairs && ok; tp += n_cl) {
      const int m0 = ((tp / p.tiles_n) * kCluster + rank) * kBM;
      const int n0 = (tp % p.tiles_n) * kBN + rank * (kBN / kCluster);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const uint32_t s = loads % kStages, use = loads / kStages;
        const bool w = bounded_wait_cl(bar(C::kEmpty + s), (use & 1u) ^ 1u, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint32_t dst = base + s * C::kStageBytes;
        const uint32_t full = mapa_shared(bar(C::kFull + s), 0);   // the leader's barrier
        if (lead) {
          if (leader) mbar_arrive_expect_tx(bar(C::kFull + s), kCluster * C::kStageBytes);
          tma_load_2d_pair(dst, &tm_x, full, kb * kBK, m0);
          tma_load_2d_pair(dst + C::kABytes, &tm_w, full, kb * kBK, n0);
        }
        ++loads;
      }
    }
    if (!ok && leader) {
      // give the copies already issued a bounded chance to land
      for (uint32_t s = 0; s < static_cast<uint32_t>(kStages) && s < loads; ++s) {
        const uint32_t n = (loads - s + kStages - 1) / kStages;  // loads into slot s
        drain_wait(bar(C::kFull + s), (n - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer (the leader CTA only) =================
    // The whole warp runs the issuer, so every operand of an MMA is
    // warp-uniform, and one elected lane issues each MMA and commit:
    // tcgen05.mma issued from a lone lane's control flow pays a large
    // per-instruction cost.
    if (leader) {
      const bool lead = elect_one();
      auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
        const bool w = bounded_wait_cl(b, parity, abort_flag, p.status);
        return __all_sync(0xffffffffu, w);
      };
      // commit to the same barrier in both CTAs of the pair
      auto commit_both = [&](uint32_t b) {
        mma_commit_pair(mapa_shared(b, 0));
        mma_commit_pair(mapa_shared(b, 1));
      };
      uint32_t uses = 0, tiles_done = 0;
      bool ok = true, issued = false;
      // descriptors advance by adding the byte offset >> 4 to the start
      // address field; every operand lies below 256 KB, so nothing carries
      const uint64_t adesc0 = sdesc_sw128(base, 16, 1024);
      const uint64_t bdesc0 = sdesc_sw128(base + C::kABytes, 16, 1024);
      for (int tp = cl; tp < p.n_pairs && ok; tp += n_cl, ++tiles_done) {
        const uint32_t buf = tiles_done & 1u, buse = tiles_done >> 1;
        if (!wait_all(bar(C::kAccEmpty + buf), (buse & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t d = tmem + buf * kBN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const uint32_t s = uses % kStages;
          // both CTAs' bytes for this slot have landed once the wait returns
          if (!wait_all(bar(C::kFull + s), (uses / kStages) & 1u)) {
            ok = false;
            break;
          }
          const uint64_t a = adesc0 + ((s * C::kStageBytes) >> 4);
          const uint64_t b = bdesc0 + ((s * C::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            if (lead)
              mma_ss_pair(d, a + ((kk * 32) >> 4), b + ((kk * 32) >> 4), C::kIdesc,
                          (kb > 0 || kk > 0) ? 1u : 0u);
          issued = true;
          // the slot is free in both CTAs once these MMAs have read it
          if (lead) commit_both(bar(C::kEmpty + s));
          ++uses;
        }
        if (!ok) break;
        if (lead) commit_both(bar(C::kAccFull + buf));
      }
      // every MMA issued so far has finished before TMEM is released
      if (issued) {
        if (lead) mma_commit_pair(mapa_shared(bar(C::kFinal), 0));
        drain_wait(bar(C::kFinal), 0, kWaitLimit);
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue: warps 2..5, TMEM lane quadrant warp % 4 =========
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t acc_empty0 = mapa_shared(bar(C::kAccEmpty), 0);   // the leader's
    uint32_t tiles_done = 0;
    for (int tp = cl; tp < p.n_pairs; tp += n_cl, ++tiles_done) {
      const uint32_t buf = tiles_done & 1u, buse = tiles_done >> 1;
      const bool ok = bounded_wait_cl(bar(C::kAccFull + buf), buse & 1u, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      fence_after_sync();
      const int m = ((tp / p.tiles_n) * kCluster + rank) * kBM + r;
      const int n0 = (tp % p.tiles_n) * kBN;
      const bool row_ok = m < p.M;
      __nv_bfloat16 *yrow = p.y + static_cast<int64_t>(row_ok ? m : 0) * p.N;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; c += 2) {
        uint32_t a0[32], a1[32];
        tmem_ld32(lane_base + buf * kBN + c * 32, a0);
        tmem_ld32(lane_base + buf * kBN + (c + 1) * 32, a1);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t *acc = h == 0 ? a0 : a1;
          const int col = n0 + (c + h) * 32;
          if (!row_ok || col >= p.N) continue;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c8 = col + 8 * v;
            if (c8 >= p.N) break;   // N is a multiple of 8
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(acc[8 * v + e]);
            if (p.bias) {
              const uint4 bv = __ldg(reinterpret_cast<const uint4 *>(p.bias + c8));
              f[0] += bf16_lo(bv.x); f[1] += bf16_hi(bv.x);
              f[2] += bf16_lo(bv.y); f[3] += bf16_hi(bv.y);
              f[4] += bf16_lo(bv.z); f[5] += bf16_hi(bv.z);
              f[6] += bf16_lo(bv.w); f[7] += bf16_hi(bv.w);
            }
            uint4 o;
            o.x = pack_bf16x2(f[0], f[1]);
            o.y = pack_bf16x2(f[2], f[3]);
            o.z = pack_bf16x2(f[4], f[5]);
            o.w = pack_bf16x2(f[6], f[7]);
            *reinterpret_cast<uint4 *>(yrow + c8) = o;
          }
        }
      }
      // every lane's TMEM reads are done; one arrival per warp on the
      // leader's barrier lets the MMA warp refill this accumulator
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty0 + 8u * buf);
    }
  }

  // ---- teardown -------------------------------------------------------------
  // neither CTA leaves while the other may still write into its shared
  // memory, arrive on its barriers or run MMAs on its TMEM
  fence_before_sync();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();
  fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// [rows, K] bf16 row-major as a 2-D tensor (K, rows); box 64 x box_rows with
// 128-byte swizzle: one K-block of box_rows rows per load.  Rows and columns
// past the end read as zero.
bool make_map_2d(CUtensorMap *map, const void *ptr, int rows, int K, int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pa

extern "C" pa_status pa_linear_bf16(const void *x, const void *w, const void *bias, void *y,
                                    int32_t M, int32_t N, int32_t K, pa_stream_t stream) {
  using namespace pa;
  if (M < 0 || N < 1 || K < 1 || !w) return PA_ERR_INVALID_ARG;
  if (M == 0) return PA_OK;   // nothing to read or write; x and y may be NULL
  if (!x || !y) return PA_ERR_INVALID_ARG;
  if ((K & 7) != 0 || (N & 7) != 0 || !aligned16(x) || !aligned16(w) || !aligned16(y) ||
      (bias && !aligned16(bias)))
    return PA_ERR_MISALIGNED;
  int32_t *status;
  int sms;
  cudaError_t e = device_context(&status, &sms);
  if (e != cudaSuccess) return from_cuda(e);
  CUtensorMap mx, mw;
  if (!make_map_2d(&mx, x, M, K, kBM) || !make_map_2d(&mw, w, N, K, kBN / kCluster))
    return from_cuda(cudaErrorInvalidValue);
  GemmParams p;
  p.bias = static_cast<const __nv_bfloat16 *>(bias);
  p.y = static_cast<__nv_bfloat16 *>(y);
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_n = (N + kBN - 1) / kBN;
  const int64_t m_pairs = ((M + kBM - 1) / kBM + kCluster - 1) / kCluster;
  const int64_t pairs = m_pairs * p.tiles_n;
  if (pairs > 0x3fffffff) return PA_ERR_UNSUPPORTED;
  p.n_pairs = static_cast<int>(pairs);
  p.k_blocks = (K + kBK - 1) / kBK;
  p.status = status;
  static unsigned long long configured = 0;
  e = set_smem_once(reinterpret_cast<const void *>(linear_bf16_kernel), GemmCfg::kSmemBytes,
                    configured);
  if (e != cudaSuccess) return from_cuda(e);
  // whole clusters, at most one CTA per SM
  const int max_ctas = sms / kCluster * kCluster;
  const int grid = kCluster * p.n_pairs < max_ctas ? kCluster * p.n_pairs : max_ctas;
  linear_bf16_kernel<<<grid, kThreads, GemmCfg::kSmemBytes,
                       reinterpret_cast<cudaStream_t>(stream)>>>(mx, mw, p);
  return from_cuda(cudaGetLastError());
}
