// C-ABI layer of libpackedattn: host-side argument checks, the per-device
// status word, and the small kernels of the packed layout (boundaries, pack,
// unpack, work order).  Attention kernels live in their own translation units.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"

namespace pa {
namespace {

// First device-side error since the last pa_get_device_status (0 = none).
__device__ int32_t g_status_word;

constexpr int kMaxDevices = 64;
int32_t *g_status_addr[kMaxDevices];
int g_num_sms[kMaxDevices];

}  // namespace

// Device address of the status word and SM count of the current device.
cudaError_t device_context(int32_t **status, int *num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (g_status_addr[dev] == nullptr) {
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_status_word);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = sms;
    g_status_addr[dev] = static_cast<int32_t *>(addr);
  }
  *status = g_status_addr[dev];
  *num_sms = g_num_sms[dev];
  return cudaSuccess;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// ---------------------------------------------------------------------------
// cu_seqlens from lengths: one CTA, chunked block scan with an int64 carry.
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    cu_seqlens_kernel(const int32_t *__restrict__ lengths, int32_t *__restrict__ cu, int batch,
                      int32_t *status) {
  __shared__ int64_t warp_sums[kScanThreads / 32];
  __shared__ int64_t carry_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry_s = 0;
    cu[0] = 0;
  }
  __syncthreads();
  bool overflow = false;
  for (int base = 0; base < batch; base += kScanThreads) {
    const int idx = base + tid;
    int64_t x = 0;
    if (idx < batch) {
      const int32_t L = lengths[idx];
      if (L < 0) record_error(status, PA_DEVICE_ERR_LENGTH);
      x = L < 0 ? 0 : L;
    }
    int64_t incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int64_t w = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = carry_s + (warp > 0 ? warp_sums[warp - 1] : 0);
    const int64_t val = before + incl;
    if (idx < batch) {
      if (val > INT32_MAX) overflow = true;
      cu[idx + 1] = static_cast<int32_t>(val > INT32_MAX ? INT32_MAX : val);
    }
    __syncthreads();
    if (tid == 0) carry_s += warp_sums[31];
    __syncthreads();
  }
  if (overflow) record_error(status, PA_DEVICE_ERR_LENGTH);
}

// ---------------------------------------------------------------------------
// pack / unpack.  The work is split into chunks of `rows_per_chunk` rows of
// one sequence (chunk c: sequence c / chunks_per_seq); a chunk's rows are
// contiguous in both layouts, so one warp copies it as one run of 16-byte
// vectors with four loads in flight per lane.  Warps stride over all chunks
// of all sequences, so a long sequence is spread over the whole GPU.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;

template <bool kPack>
__global__ void __launch_bounds__(kCopyThreads)
    repack_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                  const int32_t *__restrict__ cu, int batch, int s_max, int total,
                  int64_t row_vecs, int rows_per_chunk, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks_per_seq = (s_max + rows_per_chunk - 1) / rows_per_chunk;
  const int64_t n_chunks = chunks_per_seq * batch;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (kCopyThreads / 32);
  for (int64_t c = (static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x) >> 5;
       c < n_chunks; c += n_warps) {
    const int b = static_cast<int>(c / chunks_per_seq);
    const int64_t r0 = (c - static_cast<int64_t>(b) * chunks_per_seq) * rows_per_chunk;
    const int c0 = __ldg(cu + b), c1 = __ldg(cu + b + 1);
    const bool ok = c0 >= 0 && c0 <= c1 && c1 <= total && (b > 0 || c0 == 0);
    if (!ok || c1 - c0 > s_max) {
      if (r0 == 0 && lane == 0)
        record_error(status, ok ? PA_DEVICE_ERR_MAX_LEN : PA_DEVICE_ERR_CU_SEQLENS);
      continue;
    }
    const int64_t L = c1 - c0;
    if (r0 >= L) continue;
    const int64_t rows = L - r0 < rows_per_chunk ? L - r0 : rows_per_chunk;
    const int64_t padded_row = static_cast<int64_t>(b) * s_max + r0;
    const int64_t flat_row = static_cast<int64_t>(c0) + r0;
    const uint4 *s = src + (kPack ? padded_row : flat_row) * row_vecs;
    uint4 *d = dst + (kPack ? flat_row : padded_row) * row_vecs;
    const int64_t n = rows * row_vecs;
    int64_t i = lane;
    for (; i + 96 < n; i += 128) {
      const uint4 v0 = __ldg(s + i), v1 = __ldg(s + i + 32), v2 = __ldg(s + i + 64),
                  v3 = __ldg(s + i + 96);
      d[i] = v0;
      d[i + 32] = v1;
      d[i + 64] = v2;
      d[i + 96] = v3;
    }
    for (; i < n; i += 32) d[i] = __ldg(s + i);
  }
}

// ---------------------------------------------------------------------------
// Work order: the attention scheduler's list, written out.
// ---------------------------------------------------------------------------
constexpr int kOrderThreads = 256;

__global__ void __launch_bounds__(kOrderThreads)
    work_order_kernel(const int32_t *__restrict__ cu_q, const int32_t *__restrict__ cu_k,
                      int batch, int H, int tile_m, int32_t *__restrict__ items,
                      int64_t capacity, int32_t *status) {
  extern __shared__ int32_t sm[];
  int32_t *order = sm, *prefix = sm + batch, *tmp_lq = prefix + batch + 1,
          *tmp_lk = tmp_lq + batch;
  sched_build(order, prefix, tmp_lq, tmp_lk, cu_q, cu_k, batch, H, tile_m, INT32_MAX,
              INT32_MAX, INT32_MAX, INT32_MAX, status, true);
  const int n_items = prefix[batch];
  if (n_items > capacity && threadIdx.x == 0) record_error(status, PA_DEVICE_ERR_CAPACITY);
  const int64_t n_write = n_items < capacity ? n_items : capacity;
  for (int64_t i = threadIdx.x; i < n_write; i += kOrderThreads) {
    const WorkItem w = sched_item(order, prefix, batch, H, static_cast<int>(i));
    items[3 * i + 0] = w.seq;
    items[3 * i + 1] = w.head;
    items[3 * i + 2] = w.tile;
  }
}

// One CTA waits on an mbarrier nothing arrives at, through the same bounded
// wait the pipelined kernels use, and must come back with a timeout record.
__global__ void wait_timeout_kernel(long long limit_cycles, int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  const uint32_t b = tc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    tc::bounded_wait(b, 0, reinterpret_cast<volatile int32_t *>(&abort_flag), status,
                     limit_cycles);
}



}  // namespace

// Last CUDA error this thread saw inside the library (for pa_last_cuda_error).
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

pa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return PA_OK;
  t_last_cuda_error = e;
  return PA_ERR_CUDA;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_last_cuda_error(void) { return cudaGetErrorName(t_last_cuda_error); }

const char *pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_MISALIGNED: return "PA_ERR_MISALIGNED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
  }
  return "PA_ERR_UNKNOWN";
}

pa_status pa_varlen_attn_fwd(const void *q, const void *k, const void *v, void *out,
                             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                             int32_t batch, int32_t total_q, int32_t total_k, int32_t max_q,
                             int32_t max_k, int32_t H, int32_t D, float scale,
                             pa_stream_t stream) {
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return PA_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || max_q < 0 || max_k < 0 || H < 1 || D < 1)
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (batch > PA_MAX_BATCH || (D != 64 && D != 128) || H > 65535) return PA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k))
    return PA_ERR_MISALIGNED;
  if (total_q == 0 || max_q == 0) return PA_OK;  // no query rows: nothing to write
  VarlenArgs a{q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, max_q,
               max_k, H, D, scale, nullptr, 0};
  cudaError_t e = device_context(&a.status, &a.num_sms);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_varlen_attn(a, reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_block_window_attn_fwd(const void *q, const void *k, const void *v, void *out,
                                   int32_t batch, int32_t n, int32_t block, int32_t look_back,
                                   int32_t look_ahead, int32_t H, int32_t D, float scale,
                                   pa_stream_t stream) {
  if (!q || !k || !v || !out) return PA_ERR_INVALID_ARG;
  if (batch < 1 || n < 1 || block < 1 || look_back < 0 || look_ahead < 0 || H < 1 || D < 1)
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || H > 65535 || batch > 65535) return PA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return PA_ERR_MISALIGNED;
  BlockWindowArgs a{q, k, v, out, batch, n, block, look_back, look_ahead, H, D, scale,
                    nullptr, 0};
  cudaError_t e = device_context(&a.status, &a.num_sms);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_block_window_attn(a, reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_cu_seqlens_from_lengths(const int32_t *lengths, int32_t *cu, int32_t batch,
                                     pa_stream_t stream) {
  if (!lengths || !cu || batch < 1) return PA_ERR_INVALID_ARG;
  if (!aligned4(lengths) || !aligned4(cu)) return PA_ERR_MISALIGNED;
  int32_t *status;
  int sms;
  if (device_context(&status, &sms) != cudaSuccess) return PA_ERR_CUDA;
  cu_seqlens_kernel<<<1, kScanThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      lengths, cu, batch, status);
  return from_cuda(cudaGetLastError());
}

static pa_status repack(bool is_pack, const void *src, void *dst, const int32_t *cu,
                        int32_t batch, int32_t s_max, int32_t total, int64_t row_bytes,
                        pa_stream_t stream) {
  if (!src || !dst || !cu || batch < 1 || s_max < 0 || total < 0 || row_bytes <= 0)
    return PA_ERR_INVALID_ARG;
  if (batch > 65535) return PA_ERR_UNSUPPORTED;
  if ((row_bytes & 15) != 0 || !aligned16(src) || !aligned16(dst) || !aligned4(cu))
    return PA_ERR_MISALIGNED;
  if (s_max == 0) return PA_OK;
  int32_t *status;
  int sms;
  if (device_context(&status, &sms) != cudaSuccess) return PA_ERR_CUDA;
  // chunks of about 16 KB; a grid that fills every SM eight CTAs deep
  const int64_t vecs = row_bytes / 16;
  int64_t rows_per_chunk = 16384 / row_bytes;
  if (rows_per_chunk < 1) rows_per_chunk = 1;
  if (rows_per_chunk > s_max) rows_per_chunk = s_max;
  const int64_t n_chunks = static_cast<int64_t>(batch) * ((s_max + rows_per_chunk - 1) / rows_per_chunk);
  int64_t grid = (n_chunks + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  if (grid > static_cast<int64_t>(sms) * 8) grid = static_cast<int64_t>(sms) * 8;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  const int rpc = static_cast<int>(rows_per_chunk);
  if (is_pack)
    repack_kernel<true><<<static_cast<unsigned>(grid), kCopyThreads, 0, st>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), cu, batch, s_max, total,
        vecs, rpc, status);
  else
    repack_kernel<false><<<static_cast<unsigned>(grid), kCopyThreads, 0, st>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), cu, batch, s_max, total,
        vecs, rpc, status);
  return from_cuda(cudaGetLastError());
}

pa_status pa_pack(const void *padded, void *flat, const int32_t *cu, int32_t batch,
                  int32_t s_max, int32_t total, int64_t row_bytes, pa_stream_t stream) {
  return repack(true, padded, flat, cu, batch, s_max, total, row_bytes, stream);
}

pa_status pa_unpack(const void *flat, void *padded, const int32_t *cu, int32_t batch,
                    int32_t s_max, int32_t total, int64_t row_bytes, pa_stream_t stream) {
  return repack(false, flat, padded, cu, batch, s_max, total, row_bytes, stream);
}

int64_t pa_varlen_num_work_items(const int32_t *cu_q_host, int32_t batch, int32_t H,
                                 int32_t tile_m) {
  if (!cu_q_host || batch < 1 || H < 1 || tile_m < 1) return -1;
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = static_cast<int64_t>(cu_q_host[b + 1]) - cu_q_host[b];
    if (L < 0) return -1;
    n += static_cast<int64_t>(H) * ((L + tile_m - 1) / tile_m);
  }
  return n;
}

pa_status pa_varlen_work_order(const int32_t *cu_q, const int32_t *cu_k, int32_t batch,
                               int32_t H, int32_t tile_m, int32_t *items, int64_t capacity,
                               pa_stream_t stream) {
  if (!cu_q || !cu_k || !items || batch < 1 || H < 1 || tile_m < 1 || capacity < 0)
    return PA_ERR_INVALID_ARG;
  if (batch > PA_MAX_BATCH) return PA_ERR_UNSUPPORTED;
  if (!aligned4(cu_q) || !aligned4(cu_k) || !aligned4(items)) return PA_ERR_MISALIGNED;
  int32_t *status;
  int sms;
  if (device_context(&status, &sms) != cudaSuccess) return PA_ERR_CUDA;
  const size_t smem = sizeof(int32_t) * (4 * static_cast<size_t>(batch) + 1);
  work_order_kernel<<<1, kOrderThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      cu_q, cu_k, batch, H, tile_m, items, capacity, status);
  return from_cuda(cudaGetLastError());
}

pa_status pa_selftest_wait_timeout(int32_t timeout_us, pa_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return PA_ERR_INVALID_ARG;
  int32_t *status;
  int sms;
  if (device_context(&status, &sms) != cudaSuccess) return PA_ERR_CUDA;
  int dev = 0, khz = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  if (khz <= 0) khz = 2000000;
  const long long cycles = static_cast<long long>(timeout_us) * khz / 1000;
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(cycles, status);
  return from_cuda(cudaGetLastError());
}

pa_status pa_get_device_status(int32_t *code) {
  if (!code) return PA_ERR_INVALID_ARG;
  int32_t *status;
  int sms;
  if (device_context(&status, &sms) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  const int32_t zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return PA_ERR_CUDA;
  *code = v;
  return v == 0 ? PA_OK : PA_ERR_DEVICE;
}

}  // extern "C"
