// Temperature sampling on the device (Microgpt summary, section 推理（生成）:
// item 1 draws the next token from the predicted distribution, item 2 divides
// the logits by a temperature that sharpens or flattens it).
//
// One CTA per row. The random number is the caller's: u[b] in [0, 1) selects the
// smallest index k whose cumulative probability exceeds u[b] (inverse CDF), so a
// run is reproducible from its inputs. In fp32:
//   m = max_v l[v];  e[v] = exp((l[v] - m) / T);  Z = sum_v e[v];
// each thread owns a contiguous chunk of the row, sums its e[v], and a block scan
// turns the chunk sums into intervals [lo, hi) that tile [0, Z).
// The one thread whose interval holds u Z rescans its chunk in order and stops at
// the first index where the running sum passes u Z. Where fp32 rounding leaves
// no interval holding u Z (u Z rounded up to Z) or the running sum never passes
// it, the draw is the last index of nonzero probability, so a token of zero
// probability (a logit of -inf) is never drawn. A temperature <= 0 is the
// zero-temperature limit: the greedy index, lowest on ties.
#include <float.h>
#include <math.h>

#include <climits>

#include "common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  if (lane == 0) red[wid] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : -INFINITY;
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  return v;
}

__device__ __forceinline__ int block_max_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  if (lane == 0) red[wid] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : INT_MIN;
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  return v;
}

__device__ __forceinline__ int block_min_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  if (lane == 0) red[wid] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : INT_MAX;
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  return v;
}

// Prefix sums of one value per thread: this thread's interval [*lo, *hi) of
// [0, *total). A thread's hi and the next thread's lo are the same fp32 value (the
// same sum of the same operands), so the intervals tile [0, total) with no gap or
// overlap: within a warp both are base + (inclusive scan of the lanes before), and
// the warp bases are accumulated one after another, each equal to the previous
// base plus that warp's total.
__device__ __forceinline__ void block_intervals(float v, float* red, float* lo, float* hi,
                                                float* total) {
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  float incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const float prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 31) red[wid] = incl;   // the warp's total
  __syncthreads();
  if (threadIdx.x == 0) {
    float base = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float t = red[w];
      red[w] = base;                   // this warp's base
      base = base + t;
    }
    red[kWarps] = base;
  }
  __syncthreads();
  const float base = red[wid];
  *lo = lane == 0 ? base : base + prev;
  *hi = base + incl;
  *total = red[kWarps];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) sample_kernel(const float* __restrict__ logits, int V,
                                                          float temperature,
                                                          const float* __restrict__ u,
                                                          int32_t* __restrict__ out) {
  __shared__ float redf[kWarps + 1 > 32 ? kWarps + 1 : 32];
  __shared__ int redi[32];
  const float* row = logits + (int64_t)blockIdx.x * V;
  const int tid = threadIdx.x;
  float m = -INFINITY;
  for (int i = tid; i < V; i += kThreads) m = fmaxf(m, row[i]);
  m = block_max(m, redf);
  if (!(temperature > 0.f)) {
    // greedy: the lowest index holding the maximum
    int k = INT_MAX;
    for (int i = tid; i < V; i += kThreads)
      if (row[i] == m) {
        k = i;
        break;
      }
    k = block_min_int(k, redi);
    if (tid == 0) out[blockIdx.x] = k < V ? k : V - 1;
    return;
  }
  const float inv_t = 1.f / temperature;
  const int chunk = (V + kThreads - 1) / kThreads;
  const int c0 = min(V, tid * chunk), c1 = min(V, c0 + chunk);
  float s = 0.f;
  int last_nz = -1;   // the chunk's last index of nonzero probability
  for (int i = c0; i < c1; ++i) {
    const float e = expf((row[i] - m) * inv_t);
    s += e;
    if (e > 0.f) last_nz = i;
  }
  float lo, hi, z;
  block_intervals(s, redf, &lo, &hi, &z);
  float uu = u[blockIdx.x];
  uu = fminf(fmaxf(uu, 0.f), 0x1.fffffep-1f);   // clamp into [0, 1)
  const float target = uu * z;
  int k = INT_MAX;
  if (c0 < c1 && lo <= target && target < hi) {
    float acc = lo;
    k = last_nz;   // rounding left the running sum at or below target (hi > lo: last_nz >= c0)
    for (int i = c0; i < c1; ++i) {
      acc += expf((row[i] - m) * inv_t);
      if (acc > target) {
        k = i;
        break;
      }
    }
  }
  k = block_min_int(k, redi);
  if (k == INT_MAX) k = block_max_int(last_nz, redi);   // target rounded up to z
  if (tid == 0) out[blockIdx.x] = k >= 0 && k < V ? k : V - 1;
}

}  // namespace

void launch_sample(const float* logits, int B, int V, float temperature, const float* u,
                   int32_t* out, cudaStream_t s) {
  count_launches(1);
  sample_kernel<<<B, kThreads, 0, s>>>(logits, V, temperature, u, out);
}

}  // namespace nc
