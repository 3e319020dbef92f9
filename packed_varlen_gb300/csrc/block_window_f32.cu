// Block-window attention with fp32 inputs and outputs: the Token2Wav DiT runs
// in fp32, CFG as batch 2 ("[Perf][Model] Use block-sparse attention in
// Qwen2.5-Omni Token2Wav DiT", Purpose; its block-local result matched the
// dense masked SDPA to 6e-6, Test Result).  Query i of a batch entry sees
// key j iff j < n and -look_back <= block(j) - block(i) <= look_ahead.
//
// All arithmetic is IEEE fp32 on the CUDA cores (the tensor cores' tf32 path
// keeps 10 mantissa bits, far from the 6e-6 the fp32 model needs).  The
// layer is small and latency bound.  A CTA owns 32 query rows of one head,
// 8 per warp, and walks the union of their key windows in 32-key chunks
// staged in shared memory.  Scores: a lane per key; each lane keeps a float4
// of its K row in registers and multiplies it against the 8 rows' Q (shared
// memory broadcasts), so one K load feeds 8 rows.  The running max is
// warp-wide; the running sum stays lane-partial until the end.  P V: the
// warp's P goes through shared memory as float4 broadcasts and each lane
// owns D/32 output dimensions of all 8 rows.
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace pa {
namespace {

constexpr int kRows = 32;                 // query rows per CTA
constexpr int kWarps = 4;
constexpr int kRpw = kRows / kWarps;      // rows per warp
constexpr int kChunk = 32;                // keys per staged chunk (a lane per key)
constexpr int kThreads = kWarps * 32;

template <int D>
struct F32Smem {
  static constexpr int kKs = D + 4;       // padded K row: float4 reads hit 32 banks
  static constexpr int kQ = 0;                              // [kRows][D]
  static constexpr int kK = kQ + kRows * D;                 // [kChunk][kKs]
  static constexpr int kV = kK + kChunk * kKs;              // [kChunk][D]
  static constexpr int kP = kV + kChunk * D;                // [kWarps][kRpw][kChunk]
  static constexpr int kFloats = kP + kWarps * kRpw * kChunk;
  static constexpr int kBytes = kFloats * 4;
};

struct BwF32Params {
  const float *q, *k, *v;
  float *out;
  int64_t row_stride;  // H * D
  float scale;
  int n, block, look_back, look_ahead;
};

// [lo, hi): the keys query i may attend to.
__device__ __forceinline__ void window(const BwF32Params &p, int i, int &lo, int &hi) {
  const int64_t b = i / p.block;
  const int64_t l = (b - p.look_back) * p.block;
  const int64_t h = (b + 1 + p.look_ahead) * p.block;
  lo = static_cast<int>(l > 0 ? l : 0);
  hi = static_cast<int>(h < p.n ? h : p.n);
}

template <int D>
__global__ void __launch_bounds__(kThreads) block_window_f32_kernel(const BwF32Params p) {
  using L = F32Smem<D>;
  extern __shared__ __align__(16) float smem[];
  float *sQ = smem + L::kQ;
  float *sK = smem + L::kK;
  float *sV = smem + L::kV;
  constexpr int kPerLane = D / 32;
  constexpr int kD4 = D / 4;

  const int h = blockIdx.y, seq = blockIdx.z;
  const int r0 = blockIdx.x * kRows;
  const int n_rows = min(kRows, p.n - r0);
  const int64_t base = static_cast<int64_t>(seq) * p.n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *sP = smem + L::kP + warp * kRpw * kChunk;

  for (int idx = threadIdx.x; idx < kRows * kD4; idx += kThreads) {
    const int r = idx / kD4, d4 = idx % kD4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < n_rows)
      x = *reinterpret_cast<const float4 *>(p.q + (base + r0 + r) * p.row_stride + h * D + 4 * d4);
    *reinterpret_cast<float4 *>(sQ + r * D + 4 * d4) = x;
  }
  int k_lo, k_hi, unused;
  window(p, r0, k_lo, unused);
  window(p, r0 + n_rows - 1, unused, k_hi);

  float m[kRpw], l[kRpw], acc[kRpw][kPerLane];
  int lo[kRpw], hi[kRpw];
  int w_lo = p.n, w_hi = 0;   // union of the warp's live rows' windows
#pragma unroll
  for (int rr = 0; rr < kRpw; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int e = 0; e < kPerLane; ++e) acc[rr][e] = 0.f;
    const int r = warp * kRpw + rr;
    if (r < n_rows) {
      window(p, r0 + r, lo[rr], hi[rr]);
      w_lo = min(w_lo, lo[rr]);
      w_hi = max(w_hi, hi[rr]);
    } else {
      lo[rr] = hi[rr] = 0;   // a row past n sees no key
    }
  }

  for (int kt = k_lo; kt < k_hi; kt += kChunk) {
    __syncthreads();  // previous chunk consumed; sQ written, first time
    for (int idx = threadIdx.x; idx < kChunk * kD4; idx += kThreads) {
      const int j = idx / kD4, d4 = idx % kD4;
      float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
      if (kt + j < k_hi) {
        const int64_t off = (base + kt + j) * p.row_stride + h * D + 4 * d4;
        kk = *reinterpret_cast<const float4 *>(p.k + off);
        vv = *reinterpret_cast<const float4 *>(p.v + off);
      }
      *reinterpret_cast<float4 *>(sK + j * L::kKs + 4 * d4) = kk;
      *reinterpret_cast<float4 *>(sV + j * D + 4 * d4) = vv;
    }
    __syncthreads();
    if (w_hi <= kt || kt + kChunk <= w_lo) continue;   // warp-uniform

    float s[kRpw];
#pragma unroll
    for (int rr = 0; rr < kRpw; ++rr) s[rr] = 0.f;
    const float4 *krow = reinterpret_cast<const float4 *>(sK + lane * L::kKs);
    const float4 *qw = reinterpret_cast<const float4 *>(sQ + warp * kRpw * D);
#pragma unroll 4
    for (int d4 = 0; d4 < kD4; ++d4) {
      const float4 kk = krow[d4];
#pragma unroll
      for (int rr = 0; rr < kRpw; ++rr) {
        const float4 qq = qw[rr * kD4 + d4];
        s[rr] = fmaf(qq.x, kk.x, s[rr]);
        s[rr] = fmaf(qq.y, kk.y, s[rr]);
        s[rr] = fmaf(qq.z, kk.z, s[rr]);
        s[rr] = fmaf(qq.w, kk.w, s[rr]);
      }
    }
    const int key = kt + lane;
#pragma unroll
    for (int rr = 0; rr < kRpw; ++rr) {
      const bool ok = key >= lo[rr] && key < hi[rr];
      const float x = ok ? s[rr] * p.scale : -INFINITY;
      float cmax = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float m_new = fmaxf(m[rr], cmax);
      // no key of this row in the chunk: nothing changes
      const float alpha = m_new == -INFINITY ? 1.f : expf(m[rr] - m_new);
      const float pj = ok ? expf(x - m_new) : 0.f;
      l[rr] = l[rr] * alpha + pj;
      m[rr] = m_new;
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) acc[rr][e] *= alpha;
      sP[rr * kChunk + lane] = pj;
    }
    __syncwarp();
#pragma unroll 2
    for (int j4 = 0; j4 < kChunk / 4; ++j4) {
      float4 pp[kRpw];
#pragma unroll
      for (int rr = 0; rr < kRpw; ++rr)
        pp[rr] = *reinterpret_cast<const float4 *>(sP + rr * kChunk + 4 * j4);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float *vrow = sV + (4 * j4 + jj) * D + lane;
#pragma unroll
        for (int e = 0; e < kPerLane; ++e) {
          const float ve = vrow[32 * e];
#pragma unroll
          for (int rr = 0; rr < kRpw; ++rr) {
            const float pb = jj == 0 ? pp[rr].x : jj == 1 ? pp[rr].y : jj == 2 ? pp[rr].z : pp[rr].w;
            acc[rr][e] = fmaf(pb, ve, acc[rr][e]);
          }
        }
      }
    }
    __syncwarp();  // sP is rewritten by the next chunk
  }
#pragma unroll
  for (int rr = 0; rr < kRpw; ++rr) {
    float sum = l[rr];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const int r = warp * kRpw + rr;
    if (r >= n_rows) continue;
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    float *dst = p.out + (base + r0 + r) * p.row_stride + h * D + lane;
#pragma unroll
    for (int e = 0; e < kPerLane; ++e) dst[32 * e] = acc[rr][e] * inv;
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int D>
cudaError_t launch_f32(const BwF32Params &p, int batch, int H, cudaStream_t st) {
  static unsigned long long done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(&block_window_f32_kernel<D>),
                                F32Smem<D>::kBytes, done);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n + kRows - 1) / kRows, H, batch);
  block_window_f32_kernel<D><<<grid, kThreads, F32Smem<D>::kBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_block_window_attn_fwd_f32(const float *q, const float *k, const float *v,
                                                  float *out, int32_t batch, int32_t n,
                                                  int32_t block, int32_t look_back,
                                                  int32_t look_ahead, int32_t H, int32_t D,
                                                  float scale, pa_stream_t stream) {
  using namespace pa;
  if (!q || !k || !v || !out) return PA_ERR_INVALID_ARG;
  if (batch < 1 || n < 1 || block < 1 || look_back < 0 || look_ahead < 0 || H < 1 || D < 1)
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || H > 65535 || batch > 65535) return PA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return PA_ERR_MISALIGNED;
  BwF32Params p{q, k, v, out, static_cast<int64_t>(H) * D, scale, n, block, look_back,
                look_ahead};
  auto st = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(D == 64 ? launch_f32<64>(p, batch, H, st) : launch_f32<128>(p, batch, H, st));
}
