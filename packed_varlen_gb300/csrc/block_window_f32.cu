// Block-window attention with fp32 inputs and outputs: the Token2Wav DiT runs
// in fp32, CFG as batch 2 ("[Perf][Model] Use block-sparse attention in
// Qwen2.5-Omni Token2Wav DiT", Purpose; its block-local result matched the
// dense masked SDPA to 6e-6, Test Result).  Query i of a batch entry sees
// key j iff j < n and -look_back <= block(j) - block(i) <= look_ahead.
//
// All arithmetic is fp32 on the CUDA cores, packed two lanes wide (fma.rn
// on float2: each component rounds exactly like fmaf); the tensor cores' tf32
// path keeps 10 mantissa bits, far from the 6e-6 the fp32 model needs.  The
// softmax runs in base 2: q is scaled once by scale * log2(e), so a score is
// already a power of two and the exponentials are the hardware ex2.
//
// Work split.  Rows of one block share one key window, so a warp task is a
// run of at most kRows rows inside one block.  kSplit lanes share a group of
// kRL rows and each owns D / kSplit of their dimensions (float4 slots i with
// i % kSplit == its part).  D = 64: kSplit = 4, kRL = 3, so a task is 24
// rows, one 24-frame block on all 32 lanes (a two-lane split left 8 of 32
// lanes idle on such blocks), and each float loaded from K or V feeds three
// FMAs.  D = 128: kSplit = 2, kRL = 1, 16 rows a task.  A lane keeps its q
// slices and output accumulators in registers.  The window's keys are the
// same for the whole warp, so every K or V load is a broadcast of kSplit
// adjacent 16-byte words.  The online softmax runs per row, one update per
// stage of keys (D = 64: 12 keys, so a 24-key window takes two updates;
// D = 128: 8).  D = 128: log2(kSplit) shuffles finish a score in both lanes.
// D = 64: the row group's lanes reduce their partial scores by halves, so
// each holds 3 of the 12 scores, exponentiates only those and keeps its
// share of the row sum; the probabilities are then gathered back.  K/V stages
// hold 12 keys for D = 64 (24- and 72-key windows fill them exactly) and 16
// for D = 128.
//
// Pipeline.  Every warp is its own pipeline: it owns a run of consecutive
// tasks and streams, for each, the task's q rows and then its window in
// kStage-key K/V stages through a private kBuf-slot shared-memory ring (four
// slots for D = 64, three for D = 128: two CTAs per SM either way), so the
// next stages (and the next task's q) arrive while the current one computes.
// One lane issues each stage as TMA tensor copies (one box of q rows, or one
// box each of K and V rows) completing on the slot's mbarrier: a layer's
// loads are DRAM-bound, and per-thread 16-byte copies of these 256-byte rows
// (4 KB apart) reach only ~3.5 TB/s.  Rows outside [0, n) read as zero; V
// rows past the window in a partial last stage are cleared before use, so
// keys outside a window contribute nothing whatever their bits.  Warps never
// wait for one another.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sched.cuh"
#include "tc_ptx.cuh"
#include "tma_map.h"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

struct BwF32Params {
  float *out;
  int64_t row_stride;   // H * D
  float q_scale;        // scale * log2(e)
  int n, block, look_back, look_ahead;
  int H;
  int64_t tasks_per_row;   // tasks of one (batch entry, head): n_blocks * segs
  int n_blocks, segs;      // blocks of a sequence, tasks of a block
  int64_t n_tasks;         // over all batch entries and heads
  int tasks_per_warp;
  int32_t *status;
};

constexpr long long kWaitLimit = 4000000000LL;   // clock cycles (~2 s)
constexpr long long kDrainLimit = 400000000LL;   // teardown after an abort (~0.2 s)

// One warp task: rows [row_lo, row_hi) of batch entry `seq`, head `h`, and
// their key window [lo, hi); `off` is the element offset of (entry, row 0,
// head).
struct Task {
  int64_t off;
  int seq, h, row_lo, row_hi, lo, hi;
};

template <int D>
struct F32Shape;

// Position of a task in (batch entry, head, block, segment of the block)
// order.  A warp's tasks are consecutive, so one decode with divisions at
// the start is followed by increments only.
struct TaskPos {
  int seq, h, b, sg;
};

__device__ __forceinline__ TaskPos task_pos(const BwF32Params &p, int64_t T) {
  const int64_t rid = T / p.tasks_per_row;           // (batch entry, head)
  const int64_t t = T - rid * p.tasks_per_row;
  TaskPos c;
  c.seq = static_cast<int>(rid / p.H);
  c.h = static_cast<int>(rid - static_cast<int64_t>(c.seq) * p.H);
  c.b = static_cast<int>(t / p.segs);
  c.sg = static_cast<int>(t - static_cast<int64_t>(c.b) * p.segs);
  return c;
}

__device__ __forceinline__ void task_step(const BwF32Params &p, TaskPos &c) {
  if (++c.sg < p.segs) return;
  c.sg = 0;
  if (++c.b < p.n_blocks) return;
  c.b = 0;
  if (++c.h < p.H) return;
  c.h = 0;
  ++c.seq;
}

template <int kRows, int D>
__device__ __forceinline__ Task task_at(const BwF32Params &p, const TaskPos &c) {
  const int64_t b = c.b;
  const int64_t first = b * p.block + static_cast<int64_t>(c.sg) * kRows;
  int64_t last = first + kRows;
  if (last > (b + 1) * p.block) last = (b + 1) * p.block;
  if (last > p.n) last = p.n;
  const int64_t l = (b - p.look_back) * p.block;
  const int64_t hh = (b + 1 + p.look_ahead) * p.block;
  Task k;
  k.off = static_cast<int64_t>(c.seq) * p.n * p.row_stride + static_cast<int64_t>(c.h) * D;
  k.seq = c.seq;
  k.h = c.h;
  k.row_lo = static_cast<int>(first);
  k.row_hi = static_cast<int>(last);
  k.lo = static_cast<int>(l > 0 ? l : 0);
  k.hi = static_cast<int>(hh < p.n ? hh : p.n);
  return k;
}

template <int kStage>
__device__ __forceinline__ int kv_stages(const Task &k) {
  return (k.hi - k.lo + kStage - 1) / kStage;
}

__device__ __forceinline__ float exp2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// D = 64: four lanes share a group of three rows, 16 dimensions each, so a
// warp task is 24 rows: one 24-frame block on all 32 lanes, and every float
// loaded from K or V feeds three FMAs.  D = 128: two lanes share one row.
template <int D>
struct F32Shape {
  static constexpr int kSplit = D == 64 ? 4 : 2;    // lanes per row group
  static constexpr int kRL = D == 64 ? 3 : 1;       // rows per lane
  static constexpr int kRows = 32 / kSplit * kRL;   // rows per warp task
  static constexpr int kGroup = D == 64 ? 12 : 8;   // keys per online-softmax update
  static constexpr int kStage = D == 64 ? 12 : 16;  // keys per K/V stage (whole groups)
  static constexpr int kBuf = D == 64 ? 4 : 3;      // ring slots per warp (2 CTAs per SM)
};

template <int D>
__global__ void __launch_bounds__(kThreads)
    block_window_f32_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const BwF32Params p) {
  using S = F32Shape<D>;
  constexpr int kSplit = S::kSplit, kRL = S::kRL, kRows = S::kRows, kGroup = S::kGroup;
  constexpr int kStage = S::kStage, kBuf = S::kBuf;
  constexpr int kD4 = D / 4;                  // float4 per row
  constexpr int kF4 = kD4 / kSplit;           // float4 slots per lane and row
  constexpr int kSlot = 2 * kStage * D;       // floats per ring slot: K and V of a stage
  static_assert(kRows * D <= kSlot, "a slot holds a task's q rows");
  static_assert(kStage % kGroup == 0, "stages hold whole groups");
  extern __shared__ __align__(128) float smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *ring = smem + warp * kBuf * kSlot;
  // per warp kBuf mbarriers after all rings, then the CTA's abort flag
  const uint32_t bars = tc::smem_u32(smem + kWarps * kBuf * kSlot) + 8u * warp * kBuf;
  volatile int32_t *abort_flag =
      reinterpret_cast<volatile int32_t *>(smem + kWarps * kBuf * kSlot + 2 * kWarps * kBuf);
  if (lane == 0) {
    for (int b = 0; b < kBuf; ++b) tc::mbar_init(bars + 8u * b, 1);
    tc::fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k);
    tc::tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t t_begin = gw * p.tasks_per_warp;
  int64_t t_end = t_begin + p.tasks_per_warp;
  if (t_end > p.n_tasks) t_end = p.n_tasks;
  if (t_begin >= t_end) return;   // warps share nothing: an idle warp may leave

  // ---- producer cursor: stage `is` of task `it` (0: q rows, 1..: K/V) ----
  int64_t it = t_begin;
  int is = 0;
  TaskPos pi = task_pos(p, it);
  Task ti = task_at<kRows, D>(p, pi);
  int slot_in = 0;
  uint32_t issued = 0;   // stages issued by this warp
  auto issue_next = [&]() {
    if (it < t_end) {
      const uint32_t dst = tc::smem_u32(ring + slot_in * kSlot);
      const uint32_t bar = bars + 8u * slot_in;
      if (lane == 0) {
        // the warp's earlier reads of this slot (ordered by the __syncwarp
        // that ends every round) come before the copy's writes
        tc::fence_proxy_async();
        if (is == 0) {
          tc::mbar_arrive_expect_tx(bar, kRows * D * 4);
          tc::tma_load_4d(dst, &tm_q, bar, 0, ti.h, ti.row_lo, ti.seq);
        } else {
          const int kt = ti.lo + (is - 1) * kStage;
          tc::mbar_arrive_expect_tx(bar, 2 * kStage * D * 4);
          tc::tma_load_4d(dst, &tm_k, bar, 0, ti.h, kt, ti.seq);
          tc::tma_load_4d(dst + kStage * D * 4, &tm_v, bar, 0, ti.h, kt, ti.seq);
        }
      }
      ++issued;
      if (++is > kv_stages<kStage>(ti)) {
        is = 0;
        if (++it < t_end) {
          task_step(p, pi);
          ti = task_at<kRows, D>(p, pi);
        }
      }
    }
    slot_in = slot_in + 1 == kBuf ? 0 : slot_in + 1;
  };
#pragma unroll
  for (int s = 0; s < kBuf - 1; ++s) issue_next();

  // ---- consumer ----
  const int part = lane % kSplit;
  const int r0 = (lane / kSplit) * kRL;   // this lane's first task row
  // D = 64: the four lanes of a row group reduce their partial scores by
  // halves (a transposing butterfly), so that each ends with the full scores
  // of 3 of a group's 12 keys and computes only their exponentials; the
  // probabilities are then gathered back.  Register kk of a lane holds key
  // key_of(kk) of the group, an order that differs per lane so that every
  // exchange moves register j to register j of the partner.
  constexpr bool kTransposed = kSplit == 4 && kGroup == 12;
  const int o6 = (part & 1) ? 6 : 0, o3 = (part & 2) ? 3 : 0;
  auto key_of = [&](int kk) {
    return (kk < 6 ? o6 : 6 - o6) + (((kk / 3) & 1) ? 3 - o3 : o3) + kk % 3;
  };
  float2 q2[kRL][2 * kF4], acc2[kRL][2 * kF4];
  float m[kRL], l[kRL];
  Task tc{0, 0, 0, 0, 0, 0, 0};
  TaskPos pc = task_pos(p, t_begin);   // the consumer's current task
  int cs = 0, n_kv = 0, slot = 0;
  uint32_t consumed = 0;   // stages consumed by this warp
  bool ok = true;
  for (int64_t ct = t_begin; ct < t_end;) {
    // the stage's copies have landed (phase of the slot's consumed-th use)
    const bool w = tc::bounded_wait(bars + 8u * slot, (consumed / kBuf) & 1u, abort_flag,
                                    p.status, kWaitLimit);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    ++consumed;
    issue_next();          // refills the slot consumed last round
    float *cur = ring + slot * kSlot;
    if (cs == 0) {
      tc = task_at<kRows, D>(p, pc);
      n_kv = kv_stages<kStage>(tc);
      const float2 s2 = make_float2(p.q_scale, p.q_scale);
#pragma unroll
      for (int rr = 0; rr < kRL; ++rr) {
        const float4 *qr = reinterpret_cast<const float4 *>(cur + (r0 + rr) * D);
#pragma unroll
        for (int i = 0; i < kF4; ++i) {
          const float4 x = qr[i * kSplit + part];
          q2[rr][2 * i] = __fmul2_rn(make_float2(x.x, x.y), s2);
          q2[rr][2 * i + 1] = __fmul2_rn(make_float2(x.z, x.w), s2);
        }
#pragma unroll
        for (int i = 0; i < 2 * kF4; ++i) acc2[rr][i] = make_float2(0.f, 0.f);
        m[rr] = -INFINITY;
        l[rr] = 0.f;
      }
    } else {
      const int kt = tc.lo + (cs - 1) * kStage;
      const int e = tc.hi < kt + kStage ? tc.hi : kt + kStage;
      if (e < kt + kStage) {
        // a partial last stage: the copy brought rows past the window (or
        // zeros past n); P is 0 there, but 0 * Inf and 0 * NaN are NaN
        float4 *vz = reinterpret_cast<float4 *>(cur + kStage * D);
        for (int idx = (e - kt) * kD4 + lane; idx < kStage * kD4; idx += 32)
          vz[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
      }
      const float4 *k4 = reinterpret_cast<const float4 *>(cur) + part;
      const float4 *v4 = reinterpret_cast<const float4 *>(cur + kStage * D) + part;
#pragma unroll
      for (int g0 = 0; g0 < kStage; g0 += kGroup) {
        const int g = kt + g0;
        if (g >= e) break;   // warp-uniform
        if constexpr (kTransposed) {
          float2 sc2[kRL][kGroup];
#pragma unroll
          for (int rr = 0; rr < kRL; ++rr)
#pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) sc2[rr][kk] = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < kF4; ++i) {
#pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              const float4 kv = k4[(g0 + key_of(kk)) * kD4 + i * kSplit];
#pragma unroll
              for (int rr = 0; rr < kRL; ++rr) {
                sc2[rr][kk] = __ffma2_rn(q2[rr][2 * i], make_float2(kv.x, kv.y), sc2[rr][kk]);
                sc2[rr][kk] = __ffma2_rn(q2[rr][2 * i + 1], make_float2(kv.z, kv.w), sc2[rr][kk]);
              }
            }
          }
          // registers 6-11 go to the lane across bit 0 (where they are
          // registers 0-5, the same keys), then registers 3-5 across bit 1
          float p3[kRL][3], alpha[kRL];
#pragma unroll
          for (int rr = 0; rr < kRL; ++rr) {
            float s6[6], s3[3];
#pragma unroll
            for (int j = 0; j < 6; ++j)
              s6[j] = (sc2[rr][j].x + sc2[rr][j].y) +
                      __shfl_xor_sync(0xffffffffu, sc2[rr][j + 6].x + sc2[rr][j + 6].y, 1);
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              s3[j] = s6[j] + __shfl_xor_sync(0xffffffffu, s6[j + 3], 2);
              if (g + key_of(j) >= e) s3[j] = -INFINITY;   // keys past e: zero-filled rows
            }
            float mx = tc::fmax3(s3[0], s3[1], s3[2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m[rr], mx);   // finite: key g is in the window
            alpha[rr] = exp2_hw(m[rr] - m_new);     // 0 on the first group
            m[rr] = m_new;
#pragma unroll
            for (int j = 0; j < 3; ++j) p3[rr][j] = exp2_hw(s3[j] - m_new);
            // this lane's share of the row sum (the four are added at the end)
            l[rr] = l[rr] * alpha[rr] + (p3[rr][0] + p3[rr][1] + p3[rr][2]);
          }
          // every key's probability back into register order
          float pr[kRL][kGroup];
#pragma unroll
          for (int rr = 0; rr < kRL; ++rr) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              pr[rr][j] = p3[rr][j];
              pr[rr][j + 3] = __shfl_xor_sync(0xffffffffu, p3[rr][j], 2);
            }
#pragma unroll
            for (int j = 0; j < 6; ++j) pr[rr][j + 6] = __shfl_xor_sync(0xffffffffu, pr[rr][j], 1);
          }
#pragma unroll
          for (int i = 0; i < kF4; ++i) {
            float2 lo2[kRL], hi2[kRL];
#pragma unroll
            for (int rr = 0; rr < kRL; ++rr) {
              const float2 al2 = make_float2(alpha[rr], alpha[rr]);
              lo2[rr] = __fmul2_rn(acc2[rr][2 * i], al2);
              hi2[rr] = __fmul2_rn(acc2[rr][2 * i + 1], al2);
            }
#pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              const float4 vv = v4[(g0 + key_of(kk)) * kD4 + i * kSplit];
#pragma unroll
              for (int rr = 0; rr < kRL; ++rr) {
                const float2 pk = make_float2(pr[rr][kk], pr[rr][kk]);
                lo2[rr] = __ffma2_rn(pk, make_float2(vv.x, vv.y), lo2[rr]);
                hi2[rr] = __ffma2_rn(pk, make_float2(vv.z, vv.w), hi2[rr]);
              }
            }
#pragma unroll
            for (int rr = 0; rr < kRL; ++rr) {
              acc2[rr][2 * i] = lo2[rr];
              acc2[rr][2 * i + 1] = hi2[rr];
            }
          }
        } else {
          float2 sc2[kRL][kGroup];
  #pragma unroll
          for (int rr = 0; rr < kRL; ++rr)
  #pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) sc2[rr][kk] = make_float2(0.f, 0.f);
  #pragma unroll
          for (int i = 0; i < kF4; ++i) {
  #pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              const float4 kv = k4[(g0 + kk) * kD4 + i * kSplit];
  #pragma unroll
              for (int rr = 0; rr < kRL; ++rr) {
                sc2[rr][kk] = __ffma2_rn(q2[rr][2 * i], make_float2(kv.x, kv.y), sc2[rr][kk]);
                sc2[rr][kk] = __ffma2_rn(q2[rr][2 * i + 1], make_float2(kv.z, kv.w), sc2[rr][kk]);
              }
            }
          }
          float pr[kRL][kGroup], alpha[kRL];
  #pragma unroll
          for (int rr = 0; rr < kRL; ++rr) {
  #pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              float x = sc2[rr][kk].x + sc2[rr][kk].y;
  #pragma unroll
              for (int sh = 1; sh < kSplit; sh <<= 1) x += __shfl_xor_sync(0xffffffffu, x, sh);
              pr[rr][kk] = g + kk < e ? x : -INFINITY;   // keys past e: zero-filled rows
            }
            float mx = pr[rr][0];
  #pragma unroll
            for (int kk = 1; kk < kGroup; ++kk) mx = fmaxf(mx, pr[rr][kk]);
            const float m_new = fmaxf(m[rr], mx);       // finite: key g is in the window
            alpha[rr] = exp2_hw(m[rr] - m_new);         // 0 on the first group
            m[rr] = m_new;
            float psum = 0.f;
  #pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              pr[rr][kk] = exp2_hw(pr[rr][kk] - m_new);
              psum += pr[rr][kk];
            }
            l[rr] = l[rr] * alpha[rr] + psum;
          }
  #pragma unroll
          for (int i = 0; i < kF4; ++i) {
            float2 lo2[kRL], hi2[kRL];
  #pragma unroll
            for (int rr = 0; rr < kRL; ++rr) {
              const float2 al2 = make_float2(alpha[rr], alpha[rr]);
              lo2[rr] = __fmul2_rn(acc2[rr][2 * i], al2);
              hi2[rr] = __fmul2_rn(acc2[rr][2 * i + 1], al2);
            }
  #pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
              const float4 vv = v4[(g0 + kk) * kD4 + i * kSplit];
  #pragma unroll
              for (int rr = 0; rr < kRL; ++rr) {
                const float2 pk = make_float2(pr[rr][kk], pr[rr][kk]);
                lo2[rr] = __ffma2_rn(pk, make_float2(vv.x, vv.y), lo2[rr]);
                hi2[rr] = __ffma2_rn(pk, make_float2(vv.z, vv.w), hi2[rr]);
              }
            }
  #pragma unroll
            for (int rr = 0; rr < kRL; ++rr) {
              acc2[rr][2 * i] = lo2[rr];
              acc2[rr][2 * i + 1] = hi2[rr];
            }
          }
        }
      }
    }
    __syncwarp();   // every lane is done with this slot before it is refilled
    slot = slot + 1 == kBuf ? 0 : slot + 1;
    if (cs == n_kv) {
#pragma unroll
      for (int rr = 0; rr < kRL; ++rr) {
        const int row = tc.row_lo + r0 + rr;
        float lr = l[rr];
        if constexpr (kTransposed) {   // each lane summed its own keys
          lr += __shfl_xor_sync(0xffffffffu, lr, 1);
          lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        }
        if (row < tc.row_hi) {
          // every part of a row holds the same l
          const float inv = 1.f / lr;   // l > 0: a row always sees its own block
          float4 *dst = reinterpret_cast<float4 *>(p.out + tc.off + row * p.row_stride);
#pragma unroll
          for (int i = 0; i < kF4; ++i)
            dst[i * kSplit + part] =
                make_float4(acc2[rr][2 * i].x * inv, acc2[rr][2 * i].y * inv,
                            acc2[rr][2 * i + 1].x * inv, acc2[rr][2 * i + 1].y * inv);
        }
      }
      cs = 0;
      ++ct;
      task_step(p, pc);
    } else {
      ++cs;
    }
  }
  if (!ok) {
    // give the copies already issued a bounded chance to land
    for (uint32_t u = consumed; u < issued; ++u)
      tc::drain_wait(bars + 8u * (u % kBuf), (u / kBuf) & 1u, kDrainLimit);
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// fp32 [batch, n, H, D] as a 4-D tensor (D, H, n, batch); box D x 1 x rows
// x 1, no swizzle: `rows` consecutive tokens of one head.  Rows outside
// [0, n) of an entry read as zero.
bool make_map_f32(CUtensorMap *map, const float *ptr, int batch, int n, int H, int D, int rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(H) * D * 4,
                                 static_cast<cuuint64_t>(n) * H * D * 4};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_f32(BwF32Params p, const float *q, const float *k, const float *v, int batch,
                       int H, int sms, cudaStream_t st) {
  using S = F32Shape<D>;
  constexpr int kRows = S::kRows;
  // rings, then kBuf mbarriers per warp, then the abort flag
  constexpr int kSmem = kWarps * S::kBuf * 2 * S::kStage * D * 4 + kWarps * S::kBuf * 8 + 16;
  CUtensorMap mq, mk, mv;
  if (!make_map_f32(&mq, q, batch, p.n, H, D, kRows) ||
      !make_map_f32(&mk, k, batch, p.n, H, D, S::kStage) ||
      !make_map_f32(&mv, v, batch, p.n, H, D, S::kStage))
    return cudaErrorInvalidValue;
  static unsigned long long done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(&block_window_f32_kernel<D>),
                                kSmem, done);
  if (e != cudaSuccess) return e;
  // resident CTAs per SM, per device (a benign race: every writer stores the same value)
  static int resident[64];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int per_sm = resident[dev & 63];
  if (per_sm == 0) {
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, block_window_f32_kernel<D>,
                                                           kThreads, kSmem)) != cudaSuccess)
      return e;
    if (per_sm < 1) per_sm = 1;
    __atomic_store_n(&resident[dev & 63], per_sm, __ATOMIC_RELAXED);
  }
  const int64_t segs = (p.block + kRows - 1) / kRows;
  const int64_t n_blocks = (static_cast<int64_t>(p.n) + p.block - 1) / p.block;
  p.H = H;
  p.n_blocks = static_cast<int>(n_blocks);   // <= n
  p.segs = static_cast<int>(segs);           // <= block / kRows + 1
  p.tasks_per_row = n_blocks * segs;
  p.n_tasks = p.tasks_per_row * H * batch;
  // every warp resident at once: each takes an equal run of tasks
  const int64_t warps = static_cast<int64_t>(sms) * per_sm * kWarps;
  const int64_t tpw = (p.n_tasks + warps - 1) / warps;
  if (tpw > 0x7fffffff) return cudaErrorInvalidConfiguration;
  p.tasks_per_warp = static_cast<int>(tpw);
  const int64_t ctas = (p.n_tasks + tpw * kWarps - 1) / (tpw * kWarps);
  block_window_f32_kernel<D><<<static_cast<unsigned>(ctas), kThreads, kSmem, st>>>(mq, mk, mv, p);
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
  const float q_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (!isfinite(q_scale)) return PA_ERR_INVALID_ARG;
  int32_t *status;
  int sms;
  cudaError_t e = device_context(&status, &sms);
  if (e != cudaSuccess) return from_cuda(e);
  BwF32Params p{};
  p.out = out;
  p.row_stride = static_cast<int64_t>(H) * D;
  p.q_scale = q_scale;
  p.n = n;
  p.block = block;
  p.look_back = look_back;
  p.look_ahead = look_ahead;
  p.H = H;
  p.status = status;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(D == 64 ? launch_f32<64>(p, q, k, v, batch, H, sms, st)
                           : launch_f32<128>(p, q, k, v, batch, H, sms, st));
}
