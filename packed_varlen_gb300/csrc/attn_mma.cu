// Block-window attention of the Token2Wav DiT ("[Perf][Model] Use
// block-sparse attention in Qwen2.5-Omni Token2Wav DiT", Change): frames are
// grouped in blocks; query i sees key j iff j < n and
//   -look_back <= block(j) - block(i) <= look_ahead.
//
// The layer is small (n = 2400, H = 16, D = 64: 19.7 MB of q/k/v/out) and its
// windows are 24-72 keys wide, so it is bound by memory latency, HBM traffic
// and launch cost, not by the tensor pipe.  The kernel therefore optimises
// for memory-level parallelism: a CTA owns 64 query rows of one head and
// issues the copies of its query tile and of up to kStages 32-key K/V tiles
// of its window at once (cp.async), then runs a register-tiled flash
// attention on warp-level mma.sync (bf16 in, fp32 accumulate) with online
// softmax.  Each query row carries its own key interval [lo, hi) computed
// from the integer block parameters, so masking is two compares per score,
// no mask tensor exists, and nothing is read back from the device to decide
// whether masking applies.  A warp (16 rows, at most two 24-frame blocks)
// skips every key tile outside its rows' windows, so the scores computed
// stay close to the allowed ones.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "sched.cuh"

namespace pa {
namespace {

constexpr int kBr = 64;      // query rows per CTA: 4 warps x 16
constexpr int kBc = 32;      // keys per tile
constexpr int kThreads = 128;
constexpr int kStages = 4;   // K/V tiles in flight (a Token2Wav CTA window is <= 144 keys)

struct BwParams {
  const __nv_bfloat16 *q, *k, *v;
  __nv_bfloat16 *out;
  int64_t row_stride;  // elements between consecutive tokens (H * D)
  float scale_log2;    // scale * log2(e)
  int n, block, look_back, look_ahead;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t *>(&v);
}

// Shared tile [rows][D] bf16; 16-byte chunk c of row r lives at chunk
// c ^ (r & 7) so that ldmatrix row groups hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>((r * D + ((c ^ (r & 7)) << 3)) * 2);
}

// Copy rows [row0, row0 + kRows) of head h into a tile; rows at or beyond
// `limit` (relative to row0) are zero-filled and never read.
template <int D, int kRows>
__device__ __forceinline__ void load_tile(uint32_t dst, const __nv_bfloat16 *base, int64_t row0,
                                          int limit, int64_t stride, int h) {
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < kRows * kChunks; idx += kThreads) {
    const int r = idx / kChunks, c = idx % kChunks;
    const bool ok = r < limit;
    const __nv_bfloat16 *src = ok ? base + (row0 + r) * stride + h * D + c * 8 : base;
    cp_async16(dst + tile_off<D>(r, c), src, ok);
  }
}

// Key interval of query i: [(b - look_back) * block, (b + 1 + look_ahead) * block)
// clipped to [0, n), b = block of i.
__device__ __forceinline__ void window(const BwParams &p, int i, int &lo, int &hi) {
  const int64_t b = i / p.block;
  const int64_t l = (b - p.look_back) * p.block;
  const int64_t h = (b + 1 + p.look_ahead) * p.block;
  lo = static_cast<int>(l > 0 ? l : 0);
  hi = static_cast<int>(h < p.n ? h : p.n);
}

template <int D>
__global__ void __launch_bounds__(kThreads, D == 64 ? 4 : 2) block_window_kernel(const BwParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sK = sQ + kBr * D * 2;
  const uint32_t sV = sK + kStages * kBc * D * 2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int h = blockIdx.y;
  const int seq = blockIdx.z;

  const int q_rel0 = blockIdx.x * kBr;
  if (q_rel0 >= p.n) return;
  const int n_rows = min(kBr, p.n - q_rel0);
  const int64_t q_row0 = static_cast<int64_t>(seq) * p.n + q_rel0;
  const int64_t k_base = static_cast<int64_t>(seq) * p.n;
  int k_lo, k_hi, unused;
  window(p, q_rel0, k_lo, unused);
  window(p, q_rel0 + n_rows - 1, unused, k_hi);
  const int64_t stride = p.row_stride;
  const int ntiles = (k_hi - k_lo + kBc - 1) / kBc;

  // every copy of the first kStages tiles is issued before any wait:
  // group 0 = Q + tile 0, group s = tile s (empty groups past the window)
  load_tile<D, kBr>(sQ, p.q, q_row0, n_rows, stride, h);
  for (int s = 0; s < kStages; ++s) {
    if (s < ntiles) {
      const int kt = k_lo + s * kBc;
      load_tile<D, kBc>(sK + s * kBc * D * 2, p.k, k_base + kt, k_hi - kt, stride, h);
      load_tile<D, kBc>(sV + s * kBc * D * 2, p.v, k_base + kt, k_hi - kt, stride, h);
    }
    cp_async_commit();
  }

  // the thread's two query rows and their key intervals
  const int row_in_tile[2] = {warp * 16 + g, warp * 16 + g + 8};
  int lo[2], hi[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) window(p, q_rel0 + row_in_tile[r], lo[r], hi[r]);
  // keys any of the warp's 16 rows may see (intervals grow with the row)
  int w_lo, w_hi;
  window(p, q_rel0 + warp * 16, w_lo, unused);
  window(p, q_rel0 + warp * 16 + 15, unused, w_hi);

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  uint32_t qf[D / 16][4];

  for (int it = 0; it < ntiles; ++it) {
    const int stage = it % kStages;
    // groups 0..it are complete once at most kStages - 1 newer ones are pending
    cp_async_wait<kStages - 1>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = 2 * kk + (lane >> 4);
        ldsm_x4(sQ + tile_off<D>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const int kt = k_lo + it * kBc;
    const uint32_t tK = sK + stage * kBc * D * 2;
    const uint32_t tV = sV + stage * kBc * D * 2;
    const bool active = kt < w_hi && kt + kBc > w_lo;  // warp-uniform

    float s[kBc / 8][4];
    if (active) {
#pragma unroll
    for (int i = 0; i < kBc / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int pp = 0; pp < kBc / 16; ++pp) {
        const int r = 16 * pp + (lane & 7) + 8 * (lane >> 4);
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tK + tile_off<D>(r, c), b0, b1, b2, b3);
        mma_bf16(s[2 * pp], qf[kk], b0, b1);
        mma_bf16(s[2 * pp + 1], qf[kk], b2, b3);
      }
    }
    // scale into log2 units; keys outside the row's window -> -inf
#pragma unroll
    for (int nb = 0; nb < kBc / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kt + nb * 8 + 2 * t4 + (e & 1);
        const int r = e >> 1;
        s[nb][e] = (key >= lo[r] && key < hi[r]) ? s[nb][e] * p.scale_log2 : -INFINITY;
      }
    }
    // online softmax for the thread's two rows
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < kBc / 8; ++nb) mx = fmaxf(mx, fmaxf(s[nb][2 * r], s[nb][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[r], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_run[r] - m_use);
      m_run[r] = m_new;
      float rs = 0.f;
#pragma unroll
      for (int nb = 0; nb < kBc / 8; ++nb) {
        s[nb][2 * r] = ex2(s[nb][2 * r] - m_use);
        s[nb][2 * r + 1] = ex2(s[nb][2 * r + 1] - m_use);
        rs += s[nb][2 * r] + s[nb][2 * r + 1];
      }
      l_run[r] = l_run[r] * alpha + rs;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][2 * r] *= alpha;
        o[i][2 * r + 1] *= alpha;
      }
    }
    // O += P V
#pragma unroll
    for (int kc = 0; kc < kBc / 16; ++kc) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kc][0], s[2 * kc][1]);
      a[1] = pack_bf16(s[2 * kc][2], s[2 * kc][3]);
      a[2] = pack_bf16(s[2 * kc + 1][0], s[2 * kc + 1][1]);
      a[3] = pack_bf16(s[2 * kc + 1][2], s[2 * kc + 1][3]);
#pragma unroll
      for (int pp = 0; pp < D / 16; ++pp) {
        const int r = 16 * kc + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = 2 * pp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tV + tile_off<D>(r, c), b0, b1, b2, b3);
        mma_bf16(o[2 * pp], a, b0, b1);
        mma_bf16(o[2 * pp + 1], a, b2, b3);
      }
    }
    }  // active
    __syncthreads();  // stage `stage` is free again
    const int nxt = it + kStages;
    if (nxt < ntiles) {
      const int kn = k_lo + nxt * kBc;
      load_tile<D, kBc>(tK, p.k, k_base + kn, k_hi - kn, stride, h);
      load_tile<D, kBc>(tV, p.v, k_base + kn, k_hi - kn, stride, h);
    }
    cp_async_commit();  // (possibly empty) group keeps the group count aligned
  }
  cp_async_wait<0>();  // nothing in flight past this point

  // normalise and store the valid rows
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_run[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int row = row_in_tile[r];
    if (row < n_rows) {
      __nv_bfloat16 *dst = p.out + (q_row0 + row) * stride + h * D + 2 * t4;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        *reinterpret_cast<uint32_t *>(dst + i * 8) =
            pack_bf16(o[i][2 * r] * inv, o[i][2 * r + 1] * inv);
      }
    }
  }
}

template <int D>
cudaError_t launch_bw(const BwParams &p, dim3 grid, cudaStream_t stream) {
  const int smem = (kBr + 2 * kStages * kBc) * D * 2;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(block_window_kernel<D>), smem,
                                configured);
  if (e != cudaSuccess) return e;
  block_window_kernel<D><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_window_attn(const BlockWindowArgs &a, cudaStream_t stream) {
  BwParams p{};
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.k = static_cast<const __nv_bfloat16 *>(a.k);
  p.v = static_cast<const __nv_bfloat16 *>(a.v);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.row_stride = static_cast<int64_t>(a.H) * a.D;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.n = a.n;
  p.block = a.block;
  p.look_back = a.look_back;
  p.look_ahead = a.look_ahead;
  dim3 grid((a.n + kBr - 1) / kBr, a.H, a.batch);
  return a.D == 64 ? launch_bw<64>(p, grid, stream) : launch_bw<128>(p, grid, stream);
}

}  // namespace pa
