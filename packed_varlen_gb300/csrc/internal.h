// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed, not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "packedattn.h"

namespace pa {

// Everything an attention launch needs; filled and validated by api.cu.
struct VarlenArgs {
  const void *q, *k, *v;
  void *out;
  const int32_t *cu_q, *cu_k;
  int32_t batch, total_q, total_k, max_q, max_k, H, D;
  float scale;
  int32_t *status;  // device address of the per-device status word
  int num_sms;
};

struct BlockWindowArgs {
  const void *q, *k, *v;
  void *out;
  int32_t batch, n, block, look_back, look_ahead, H, D;
  float scale;
  int32_t *status;
  int num_sms;
};

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute persists; setting it on every launch costs host time between
// back-to-back launches).  `done` is the caller's per-kernel device bitmask.
inline cudaError_t set_smem_once(const void *kernel, int smem, unsigned long long &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) __atomic_fetch_or(&done, bit, __ATOMIC_ACQ_REL);
  return e;
}

// Device address of the per-device status word and the SM count of the
// current device (api.cu).
cudaError_t device_context(int32_t **status, int *num_sms);

// Maps a CUDA error to a pa_status and remembers it for pa_last_cuda_error.
pa_status from_cuda(cudaError_t e);

// Launchers: return cudaSuccess or the launch error.
cudaError_t launch_varlen_attn(const VarlenArgs &a, cudaStream_t stream);
cudaError_t launch_varlen_attn_pair(const VarlenArgs &a, cudaStream_t stream);   // D = 128
cudaError_t launch_block_window_attn(const BlockWindowArgs &a, cudaStream_t stream);

}  // namespace pa
