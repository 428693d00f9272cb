// Next-token loss of the training step (Microgpt summary, section 训练过程, item 2:
// the cross-entropy between the predicted distribution and the true next token),
// finished from the LM head's per-block softmax partials. The LM-head GEMM's
// epilogue reduces each 256-column block of a row to (m, s) = (max z, sum
// exp(z - m)) and keeps the target's logit, so the logits themselves are never
// stored. Here one warp per row merges its blocks,
//   M = max m_nb,  S = sum s_nb exp(m_nb - M),  loss = log S + M - z_target,
// and one block sums the rows' losses in a fixed order for the mean.
#include <math.h>

#include "common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

// One warp per row: lane j merges blocks j, j + 32, ... in order, then the
// lanes' pairs are merged by a butterfly (max first, then the rescaled sums).
__global__ void ce_rows_kernel(const float2* __restrict__ part, int nblk, int64_t M,
                               const float* __restrict__ zt, const int32_t* __restrict__ targets,
                               int V, float* __restrict__ loss, uint32_t* status) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (r >= M) return;   // uniform across the warp
  const int t = targets[r];
  if (t < 0 || t >= V) {
    if (lane == 0) {
      loss[r] = 0.f;
      if (t >= V && status) atomicOr(status, ST_BAD_TOKEN);
    }
    return;
  }
  float mx = -INFINITY, S = 0.f;
  for (int nb = lane; nb < nblk; nb += 32) {
    const float2 q = part[(int64_t)nb * M + r];
    if (q.x > mx) {
      S = S * expf(mx - q.x) + q.y;   // S is 0 while mx is -inf
      mx = q.x;
    } else {
      S += q.y * expf(q.x - mx);
    }
  }
  float gm = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
  S = mx > -INFINITY ? S * expf(mx - gm) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  if (lane == 0) loss[r] = logf(S) + gm - zt[r];
}

constexpr int kMeanThreads = 1024;

// Sum of the counted rows' losses, in double: thread i adds rows i, i + 1024, ...
// in order, then a fixed tree over the threads.
__global__ void __launch_bounds__(kMeanThreads)
    ce_mean_kernel(const float* __restrict__ loss, const int32_t* __restrict__ targets, int V,
                   int64_t M, float* mean) {
  __shared__ double ssum[kMeanThreads];
  __shared__ long long scnt[kMeanThreads];
  double a = 0.0;
  long long n = 0;
  for (int64_t r = threadIdx.x; r < M; r += kMeanThreads) {
    const int t = targets[r];
    if (t >= 0 && t < V) {
      a += (double)loss[r];
      ++n;
    }
  }
  ssum[threadIdx.x] = a;
  scnt[threadIdx.x] = n;
  __syncthreads();
  for (int w = kMeanThreads / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) {
      ssum[threadIdx.x] += ssum[threadIdx.x + w];
      scnt[threadIdx.x] += scnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *mean = scnt[0] ? (float)(ssum[0] / (double)scnt[0]) : __int_as_float(0x7fc00000);
}

}  // namespace

void launch_ce_finish(const float2* part, int nblk, const float* zt, const int32_t* targets,
                      int V, int64_t M, float* loss, float* mean, uint32_t* status,
                      cudaStream_t s) {
  if (M > 0)
    ce_rows_kernel<<<(unsigned)((M + 7) / 8), 256, 0, s>>>(part, nblk, M, zt, targets, V, loss,
                                                           status);
  ce_mean_kernel<<<1, kMeanThreads, 0, s>>>(loss, targets, V, M, mean);
  count_launches(M > 0 ? 2 : 1);
}

}  // namespace nc
