// Rotary position embedding on packed q and k with request-local positions.
//
// The dynamic path rebuilds RoPE per request from request-local state and
// never infers positions from packed global offsets ("feat: Support dynamic
// batching for heterogeneous diffusion requests", Correctness model; the
// packed path's RoPE runs as one fused operator, "[Perf][Diffusion]
// [Qwen-Image] Replace per-bucket varlen loop ...").  Token j of packed
// sequence b sits at position p = pos_offset[b] + j; every head's interleaved
// pairs (x_2i, x_2i+1) are rotated by p * base^(-2i/D).
//
// HBM bound (q and k read and written once, in place).  One warp per token
// row: the warp builds the row's D/2 (cos, sin) pairs once in shared memory
// and applies them to all H heads with 16-byte vector loads and stores.  The
// angle is reduced exactly: the fraction of a turn, p * theta_i / (2 pi), is
// taken in double precision, then sincospif gives sin and cos in fp32.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sched.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;     // 8 warps, one token row each per step
constexpr int kMaxHalfD = 256;    // D <= 512

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads)
    rope_kernel(__nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ k,
                const int32_t *__restrict__ cu_q, const int32_t *__restrict__ cu_k,
                const int32_t *__restrict__ pos_offset, int total_q, int total_k, int H,
                int D, double log2_base, int32_t *status) {
  __shared__ double turns_per_pos[kMaxHalfD];   // theta_i / (2 pi)
  __shared__ float2 cs[kThreads / 32][kMaxHalfD];
  const int half = D / 2;
  for (int i = threadIdx.x; i < half; i += kThreads)
    turns_per_pos[i] = exp2(-2.0 * i / D * log2_base) * 0.15915494309189535;  // / (2 pi)
  __syncthreads();

  const int b = blockIdx.y;
  const bool is_k = blockIdx.z == 1;
  const int32_t *cu = is_k ? cu_k : cu_q;
  __nv_bfloat16 *x = is_k ? k : q;
  const int total = is_k ? total_k : total_q;
  const int c0 = __ldg(cu + b), c1 = __ldg(cu + b + 1);
  if (c0 < 0 || c0 > c1 || c1 > total || (b == 0 && c0 != 0)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, PA_DEVICE_ERR_CU_SEQLENS);
    return;
  }
  const int off = pos_offset ? __ldg(pos_offset + b) : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_vecs = H * D / 8;
  const int head_vecs = D / 8;
  for (int j = blockIdx.x * (kThreads / 32) + warp; j < c1 - c0;
       j += gridDim.x * (kThreads / 32)) {
    const double p = static_cast<double>(off) + j;
    for (int i = lane; i < half; i += 32) {
      double t = p * turns_per_pos[i];
      t -= floor(t);
      float sn, cn;
      sincospif(2.f * static_cast<float>(t), &sn, &cn);
      cs[warp][i] = make_float2(cn, sn);
    }
    __syncwarp();
    uint4 *row = reinterpret_cast<uint4 *>(x + static_cast<int64_t>(c0 + j) * H * D);
    for (int v = lane; v < row_vecs; v += 32) {
      const int i0 = (v % head_vecs) * 4;   // first pair of this 8-element vector
      float a[8];
      bf16x8_to_f32(row[v], a);
      float o[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 c = cs[warp][i0 + m];
        o[2 * m] = a[2 * m] * c.x - a[2 * m + 1] * c.y;
        o[2 * m + 1] = a[2 * m] * c.y + a[2 * m + 1] * c.x;
      }
      uint4 w;
      w.x = pack2(o[0], o[1]);
      w.y = pack2(o[2], o[3]);
      w.z = pack2(o[4], o[5]);
      w.w = pack2(o[6], o[7]);
      row[v] = w;
    }
    __syncwarp();
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace pa

extern "C" pa_status pa_rope_packed(void *q, void *k, const int32_t *cu_seqlens_q,
                                    const int32_t *cu_seqlens_k, const int32_t *pos_offset,
                                    int32_t batch, int32_t total_q, int32_t total_k,
                                    int32_t H, int32_t D, float base, pa_stream_t stream) {
  using namespace pa;
  if (!q || !k || !cu_seqlens_q || !cu_seqlens_k) return PA_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || H < 1 || D < 2 || (D & 1))
    return PA_ERR_INVALID_ARG;
  if (!isfinite(base) || !(base > 0.f)) return PA_ERR_INVALID_ARG;
  if (batch > 65535 || D > 2 * kMaxHalfD || (D & 7)) return PA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k) ||
      (pos_offset && !aligned4(pos_offset)))
    return PA_ERR_MISALIGNED;
  int32_t *status;
  int sms;
  cudaError_t e = device_context(&status, &sms);
  if (e != cudaSuccess) return from_cuda(e);
  const int longest = total_q > total_k ? total_q : total_k;
  if (longest == 0) return PA_OK;
  int per_seq = (sms * 8 + batch - 1) / batch;
  const int max_blocks = (longest + kThreads / 32 - 1) / (kThreads / 32);
  if (per_seq > max_blocks) per_seq = max_blocks;
  if (per_seq < 1) per_seq = 1;
  dim3 grid(per_seq, batch, 2);
  rope_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<__nv_bfloat16 *>(q), static_cast<__nv_bfloat16 *>(k), cu_seqlens_q,
      cu_seqlens_k, pos_offset, total_q, total_k, H, D, log2(static_cast<double>(base)), status);
  return from_cuda(cudaGetLastError());
}
