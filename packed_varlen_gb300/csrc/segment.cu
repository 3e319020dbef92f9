// Segment-aware unpack with the per-request classifier-free-guidance combine
// ("feat: Support dynamic batching for heterogeneous diffusion requests",
// AttentionSegment and CFG behavior):
//   out[r, i, :] = neg_i + true_cfg_scale[r] * (pos_i - neg_i)
// over the image span of request r's positive and negative packed sequences,
// optionally rescaled to the positive row's L2 norm (cfg_normalize).
//
// HBM bound: one warp per output row (several rows per warp when a row has
// fewer than 32 sixteen-byte vectors), 16-byte vector loads and stores with
// four vectors of each input in flight per lane, fp32 arithmetic (one fused
// multiply-add per element), bf16 round to nearest.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sched.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;  // 8 warps, one output row each per step
constexpr int kBatch = 4;      // 16-byte vectors per lane and input in flight

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

struct Span {
  int64_t pos0, neg0;  // first image row of the positive / negative sequence
  int n_img;           // image rows (-1: invalid request)
};

__device__ Span request_span(const int32_t *__restrict__ cu, const int32_t *__restrict__ img_off,
                             int p, int q, int batch, int total, int img_max) {
  Span sp{0, 0, -1};
  auto seq = [&](int b, int64_t &first, int &n) -> bool {
    if (b < 0 || b >= batch) return false;
    const int c0 = __ldg(cu + b), c1 = __ldg(cu + b + 1), off = __ldg(img_off + b);
    if (c0 < 0 || c0 > c1 || c1 > total || off < 0 || off > c1 - c0) return false;
    first = static_cast<int64_t>(c0) + off;
    n = c1 - c0 - off;
    return true;
  };
  int np = 0, nq = 0;
  if (!seq(p, sp.pos0, np)) return sp;
  if (q >= 0 && (!seq(q, sp.neg0, nq) || nq != np)) return sp;
  if (np > img_max) return sp;
  sp.n_img = np;
  return sp;
}

__global__ void __launch_bounds__(kThreads)
    cfg_combine_kernel(const __nv_bfloat16 *__restrict__ flat, __nv_bfloat16 *__restrict__ out,
                       const int32_t *__restrict__ cu, const int32_t *__restrict__ img_off,
                       const int32_t *__restrict__ pos_seq, const int32_t *__restrict__ neg_seq,
                       const float *__restrict__ cfg_scale,
                       const int32_t *__restrict__ cfg_normalize, int batch, int total,
                       int img_max, int row_elems, int32_t *status) {
  const int r = blockIdx.y;
  const int p = __ldg(pos_seq + r), q = __ldg(neg_seq + r);
  const Span sp = request_span(cu, img_off, p, q, batch, total, img_max);
  if (sp.n_img < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, PA_DEVICE_ERR_SEGMENT);
    return;
  }
  const bool cfg = q >= 0;
  const float s = cfg ? __ldg(cfg_scale + r) : 1.f;
  const bool normalize = cfg && __ldg(cfg_normalize + r) != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vecs = row_elems / 8;
  // narrow rows (a power-of-two count of 16-byte vectors below 32): several
  // rows per warp, `group` lanes each; wide rows: one row per warp
  const int group = (vecs < 32 && (vecs & (vecs - 1)) == 0) ? vecs : 32;
  const int rows_per_warp = 32 / group;
  const int sub = lane / group, gl = lane % group;
  const int rows_per_step = (kThreads / 32) * rows_per_warp;
  for (int i0 = blockIdx.x * rows_per_step; i0 < sp.n_img; i0 += gridDim.x * rows_per_step) {
    const int i = i0 + warp * rows_per_warp + sub;
    const bool live = i < sp.n_img;   // uniform within a lane group
    const uint4 *pr = reinterpret_cast<const uint4 *>(flat + (sp.pos0 + i) * row_elems);
    const uint4 *nr = reinterpret_cast<const uint4 *>(flat + (sp.neg0 + i) * row_elems);
    uint4 *orow = reinterpret_cast<uint4 *>(out + (static_cast<int64_t>(r) * img_max + i) * row_elems);
    float factor = 1.f;
    if (normalize) {
      // pass 1: squared norms of the positive and the combined row
      float pp = 0.f, cc = 0.f;
      if (live) {
        for (int v = gl; v < vecs; v += group) {
          float a[8], b[8];
          bf16x8_to_f32(__ldg(pr + v), a);
          bf16x8_to_f32(__ldg(nr + v), b);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float c = fmaf(s, a[k] - b[k], b[k]);
            pp = fmaf(a[k], a[k], pp);
            cc = fmaf(c, c, cc);
          }
        }
      }
      // reduce within the lane group (offsets below the group width)
      for (int off = group >> 1; off > 0; off >>= 1) {
        pp += __shfl_xor_sync(0xffffffffu, pp, off);
        cc += __shfl_xor_sync(0xffffffffu, cc, off);
      }
      factor = cc > 0.f ? sqrtf(pp) / sqrtf(cc) : 0.f;
    }
    if (!live) continue;
    // kBatch vectors of each input per lane loaded before any is combined
    for (int v0 = gl; v0 < vecs; v0 += group * kBatch) {
      uint4 ain[kBatch], bin[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int v = v0 + group * u;
        if (v < vecs) {
          ain[u] = __ldg(pr + v);
          if (cfg) bin[u] = __ldg(nr + v);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int v = v0 + group * u;
        if (v >= vecs) break;
        float a[8];
        bf16x8_to_f32(ain[u], a);
        float c[8];
        if (cfg) {
          float b[8];
          bf16x8_to_f32(bin[u], b);
#pragma unroll
          for (int k = 0; k < 8; ++k) c[k] = fmaf(s, a[k] - b[k], b[k]) * factor;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) c[k] = a[k];
        }
        uint4 w;
        w.x = pack2(c[0], c[1]);
        w.y = pack2(c[2], c[3]);
        w.z = pack2(c[4], c[5]);
        w.w = pack2(c[6], c[7]);
        orow[v] = w;
      }
    }
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace pa

extern "C" pa_status pa_cfg_combine(const void *flat, void *out, const int32_t *cu,
                                    const int32_t *img_off, const int32_t *pos_seq,
                                    const int32_t *neg_seq, const float *cfg_scale,
                                    const int32_t *cfg_normalize, int32_t batch,
                                    int32_t requests, int32_t total, int32_t img_max,
                                    int32_t row_elems, pa_stream_t stream) {
  using namespace pa;
  if (!flat || !out || !cu || !img_off || !pos_seq || !neg_seq || !cfg_scale || !cfg_normalize)
    return PA_ERR_INVALID_ARG;
  if (batch < 1 || requests < 1 || total < 0 || img_max < 0 || row_elems < 1)
    return PA_ERR_INVALID_ARG;
  if (batch > 65535 || requests > 65535) return PA_ERR_UNSUPPORTED;
  if ((row_elems & 7) != 0 || !aligned16(flat) || !aligned16(out) || !aligned4(cu) ||
      !aligned4(img_off) || !aligned4(pos_seq) || !aligned4(neg_seq) || !aligned4(cfg_scale) ||
      !aligned4(cfg_normalize))
    return PA_ERR_MISALIGNED;
  if (img_max == 0) return PA_OK;
  int32_t *status;
  int sms;
  cudaError_t e = device_context(&status, &sms);
  if (e != cudaSuccess) return from_cuda(e);
  // enough warps to cover the GPU a few times over all requests
  const int vecs = row_elems / 8;
  const int rows_per_block =
      (kThreads / 32) * ((vecs < 32 && (vecs & (vecs - 1)) == 0) ? 32 / vecs : 1);
  int per_req = (sms * 16 + requests - 1) / requests;
  const int max_blocks = (img_max + rows_per_block - 1) / rows_per_block;
  if (per_req > max_blocks) per_req = max_blocks;
  if (per_req < 1) per_req = 1;
  dim3 grid(per_req, requests);
  cfg_combine_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(flat), static_cast<__nv_bfloat16 *>(out), cu, img_off,
      pos_seq, neg_seq, cfg_scale, cfg_normalize, batch, total, img_max, row_elems, status);
  return from_cuda(cudaGetLastError());
}
