// CUDA-core kernels: embedding + norm, RMSNorm, the fp32 GEMM, projection
// epilogues applied after split-K reductions, fp32 attention, argmax.
#include <float.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "nc_internal.h"

namespace nc {

// ---------------------------------------------------------------- row helpers
template <class T> struct Vec4 {   // 16-bit types: 8-byte accesses
  __device__ static float4 load(const T* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    float2 fa = unpack2<T>(u.x), fb = unpack2<T>(u.y);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
  }
  __device__ static void store(T* p, float4 v) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack2<T>(v.x, v.y), pack2<T>(v.z, v.w));
  }
};
template <> struct Vec4<float> {
  __device__ static float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  __device__ static void store(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};

// Embedding row gather (RMSNorm of the block-1 input fused in): one warp per
// token row. x = wte[tok] in fp32; xn = x / sqrt(mean x^2 + eps) in T.
template <class TW, class T>
__global__ void embed_norm_kernel(const int32_t* __restrict__ tok, const TW* __restrict__ wte,
                                  float* __restrict__ x, T* __restrict__ xn, int64_t M, int d,
                                  int vocab, float eps, uint32_t* status) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= M) return;
  int id = tok[row];
  if (id < 0 || id >= vocab) {
    if (lane == 0) atomicOr(status, ST_BAD_TOKEN);
    id = 0;
  }
  const TW* src = wte + (int64_t)id * d;
  float* xr = x + row * d;
  float ss = 0.f;
  for (int j = lane * 4; j < d; j += 128) {
    float4 v = Vec4<TW>::load(src + j);
    Vec4<float>::store(xr + j, v);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / d + eps);
  T* yr = xn + row * d;
  for (int j = lane * 4; j < d; j += 128) {
    float4 v = Vec4<float>::load(xr + j);
    Vec4<T>::store(yr + j, make_float4(v.x * r, v.y * r, v.z * r, v.w * r));
  }
}

// RMSNorm without gain, one warp per row, 16-byte loads.
template <class T>
__global__ void rmsnorm_kernel(const float* __restrict__ x, T* __restrict__ y, int64_t M, int d,
                               float eps) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= M) return;
  const float* xr = x + row * d;
  float ss = 0.f;
  for (int j = lane * 4; j < d; j += 128) {
    float4 v = Vec4<float>::load(xr + j);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / d + eps);
  T* yr = y + row * d;
  for (int j = lane * 4; j < d; j += 128) {
    float4 v = Vec4<float>::load(xr + j);
    Vec4<T>::store(yr + j, make_float4(v.x * r, v.y * r, v.z * r, v.w * r));
  }
}

// ---------------------------------------------------------------- fp32 GEMM
// C[M, N] = A[M, K] B[N, K]^T with fp32 accumulation; 64x64 tile per block of
// 256 threads, 4x4 outputs per thread, K staged 16 at a time through shared memory.
template <class T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ A,
                                                        const T* __restrict__ B,
                                                        float* __restrict__ C, int64_t M, int N,
                                                        int K, int64_t ldc) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * 64;
  const int n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, c = i % 16;
      const int64_t m = m0 + r;
      const int n = n0 + r, k = k0 + c;
      As[c][r] = (m < M && k < K) ? to_f32(A[m * K + k]) : 0.f;
      Bs[c][r] = (n < N && k < K) ? to_f32(B[(int64_t)n * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) C[m * ldc + n] = acc[i][j];
    }
  }
}

// ----------------------------------------------------- projection epilogues
// Q/K/V epilogue: sums the split-K partials of one (row, head), applies RoPE to
// Q and K heads (pairs (i, i + hd/2) rotated by +theta(t, i)), then the QK RMS
// norm, and scatters: Q -> q[b][h][t - pos0], K -> k_cache[b][g][t], V (as
// projected) -> v_cache[b][g][t]. One warp per (row, head); lane owns pairs
// i = lane + 32 r.
template <class T>
__global__ void qkv_post_kernel(const float* __restrict__ part, int n_split, int64_t M,
                                RowMap rm, QkvDst dst) {
  const int heads = dst.H + 2 * dst.Hkv;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (w >= M * heads) return;
  const int64_t row = w / heads;
  const int j = (int)(w % heads);
  const int hd = dst.hd, half = hd / 2;
  const int N = heads * hd;
  const int b = (int)(row / rm.rows_per_seq);
  const int t = rm.pos0 + (int)(row % rm.rows_per_seq);
  const int64_t split_stride = M * N;
  float lo[4], hi[4];
  int cnt = 0;
  float ss = 0.f;
  for (int i = lane; i < half; i += 32, ++cnt) {
    float a = 0.f, c = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float* p = part + s * split_stride + row * N + (int64_t)j * hd;
      a += p[i];
      c += p[i + half];
    }
    lo[cnt] = a;
    hi[cnt] = c;
  }
  if (j >= dst.H + dst.Hkv) {  // V head: stored as projected
    const int g = j - dst.H - dst.Hkv;
    T* out = reinterpret_cast<T*>(dst.v_cache) + (((int64_t)b * dst.Hkv + g) * dst.t_max + t) * hd;
    cnt = 0;
    float amax = 0.f;
    for (int i = lane; i < half; i += 32, ++cnt) {
      out[i] = from_f32<T>(lo[cnt]);
      out[i + half] = from_f32<T>(hi[cnt]);
      amax = fmaxf(amax, fmaxf(fabsf(lo[cnt]), fabsf(hi[cnt])));
    }
    note_range<T>(amax, dst.status);
    return;
  }
  cnt = 0;
  for (int i = lane; i < half; i += 32, ++cnt) {
    const float cs = dst.cos_tab[(int64_t)t * half + i], sn = dst.sin_tab[(int64_t)t * half + i];
    const float a = lo[cnt], c = hi[cnt];
    lo[cnt] = a * cs - c * sn;
    hi[cnt] = a * sn + c * cs;
    ss += lo[cnt] * lo[cnt] + hi[cnt] * hi[cnt];
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / hd + dst.eps);
  T* out;
  if (j < dst.H) {
    out = reinterpret_cast<T*>(dst.q) +
          (((int64_t)b * dst.H + j) * rm.rows_per_seq + (t - rm.pos0)) * hd;
  } else {
    const int g = j - dst.H;
    out = reinterpret_cast<T*>(dst.k_cache) + (((int64_t)b * dst.Hkv + g) * dst.t_max + t) * hd;
  }
  cnt = 0;
  for (int i = lane; i < half; i += 32, ++cnt) {
    out[i] = from_f32<T>(lo[cnt] * r);
    out[i + half] = from_f32<T>(hi[cnt] * r);
  }
}

// x[m, :] += sum of partials; optionally writes RMSNorm(x[m, :]) to xn. One warp per row.
template <class T>
__global__ void residual_finish_kernel(const float* __restrict__ part, int n_split,
                                       float* __restrict__ x, int64_t M, int N,
                                       T* __restrict__ xn, float eps) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= M) return;
  float* xr = x + row * N;
  float ss = 0.f;
  for (int j = lane * 4; j < N; j += 128) {
    float4 v = Vec4<float>::load(xr + j);
    for (int s = 0; s < n_split; ++s) {
      float4 p = Vec4<float>::load(part + s * M * N + row * N + j);
      v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
    }
    Vec4<float>::store(xr + j, v);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (xn == nullptr) return;
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / N + eps);
  T* yr = xn + row * N;
  for (int j = lane * 4; j < N; j += 128) {
    float4 v = Vec4<float>::load(xr + j);
    Vec4<T>::store(yr + j, make_float4(v.x * r, v.y * r, v.z * r, v.w * r));
  }
}

// h = relu(sum of partials)^2, elementwise.
template <class T>
__global__ void relu2_finish_kernel(const float* __restrict__ part, int n_split,
                                    T* __restrict__ h, int64_t total, uint32_t* status) {
  float amax = 0.f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < n_split; ++s) a += part[s * total + i];
    a = fmaxf(a, 0.f);
    amax = fmaxf(amax, a * a);
    h[i] = from_f32<T>(a * a);
  }
  note_range<T>(amax, status);
}

__global__ void sum_splits_kernel(const float* __restrict__ part, int n_split,
                                  float* __restrict__ out, int64_t M, int N, int64_t ldo) {
  const int64_t total = M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < n_split; ++s) a += part[s * total + i];
    out[(i / N) * ldo + i % N] = a;
  }
}

// ----------------------------------------------------------- fp32 attention
// One warp per query. Keys are visited 32 at a time (one per lane for the
// score), then the value accumulation runs with lanes over head dimensions.
// Online softmax: running max m, running sum l, unnormalised accumulator o.
// Writes the normalised output, or (for split decode) the raw (m, l, o).
template <class T>
__device__ void attend_one_query(const T* __restrict__ qv, const T* __restrict__ kb,
                                 const T* __restrict__ vb, int s_begin, int s_end, int hd,
                                 float scale, float* q_sh, float& m_run, float& l_run,
                                 float (&o)[4]) {
  const int lane = threadIdx.x % 32;
  for (int i = lane; i < hd; i += 32) q_sh[i] = to_f32(qv[i]);
  __syncwarp();
  for (int s0 = s_begin; s0 < s_end; s0 += 32) {
    const int s = s0 + lane;
    float sc = -INFINITY;
    if (s < s_end) {
      const T* kr = kb + (int64_t)s * hd;
      float acc = 0.f;
      for (int i = 0; i < hd; ++i) acc = fmaf(q_sh[i], to_f32(kr[i]), acc);
      sc = acc * scale;
    }
    const float m_new = fmaxf(m_run, warp_max(sc));
    const float p = (s < s_end) ? __expf(sc - m_new) : 0.f;
    const float corr = __expf(m_run - m_new);
    l_run = l_run * corr + warp_sum(p);
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] *= corr;
    const int n = min(32, s_end - s0);
    for (int u = 0; u < n; ++u) {
      const float pu = __shfl_sync(0xffffffffu, p, u);
      const T* vr = vb + (int64_t)(s0 + u) * hd;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = lane + 32 * r;
        if (i < hd) o[r] = fmaf(pu, to_f32(vr[i]), o[r]);
      }
    }
    m_run = m_new;
  }
}

template <class T>
__global__ void attention_prefill_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                              const T* __restrict__ v, T* __restrict__ o, int B,
                                              int H, int Hkv, int T_, int t_max, int hd) {
  extern __shared__ float q_smem[];
  const int warps = blockDim.x / 32;
  const int64_t w = (int64_t)blockIdx.x * warps + threadIdx.x / 32;
  if (w >= (int64_t)B * H * T_) return;
  const int t = (int)(w % T_);
  const int h = (int)((w / T_) % H);
  const int b = (int)(w / ((int64_t)T_ * H));
  const int g = h / (H / Hkv);
  float* q_sh = q_smem + (threadIdx.x / 32) * hd;
  const T* qv = q + (((int64_t)b * H + h) * T_ + t) * hd;
  const T* kb = k + ((int64_t)b * Hkv + g) * t_max * hd;
  const T* vb = v + ((int64_t)b * Hkv + g) * t_max * hd;
  float m_run = -INFINITY, l_run = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  attend_one_query(qv, kb, vb, 0, t + 1, hd, rsqrtf((float)hd), q_sh, m_run, l_run, acc);
  const int lane = threadIdx.x % 32;
  T* out = o + ((int64_t)b * T_ + t) * H * hd + (int64_t)h * hd;
  const float inv = 1.f / l_run;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = lane + 32 * r;
    if (i < hd) out[i] = from_f32<T>(acc[r] * inv);
  }
}

// Split decode: block (b*H + h, split). scratch layout per (b, h, split):
// [m, l, o[hd]] fp32.
template <class T>
__global__ void attention_decode_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                             const T* __restrict__ v, float* __restrict__ scratch,
                                             int B, int H, int Hkv, int len, int t_max, int hd,
                                             int n_split) {
  extern __shared__ float q_smem[];
  const int bh = blockIdx.x;
  const int split = blockIdx.y;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / Hkv);
  const int chunk = (len + n_split - 1) / n_split;
  const int s_begin = split * chunk, s_end = min(len, s_begin + chunk);
  float m_run = -INFINITY, l_run = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  const T* kb = k + ((int64_t)b * Hkv + g) * t_max * hd;
  const T* vb = v + ((int64_t)b * Hkv + g) * t_max * hd;
  if (s_begin < s_end)
    attend_one_query(q + (int64_t)bh * hd, kb, vb, s_begin, s_end, hd, rsqrtf((float)hd), q_smem,
                     m_run, l_run, acc);
  float* rec = scratch + ((int64_t)bh * n_split + split) * (hd + 2);
  const int lane = threadIdx.x % 32;
  if (lane == 0) {
    rec[0] = m_run;
    rec[1] = l_run;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = lane + 32 * r;
    if (i < hd) rec[2 + i] = acc[r];
  }
}

// Log-sum-exp merge of the split states: o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
template <class T>
__global__ void attention_combine_kernel(const float* __restrict__ scratch, T* __restrict__ o,
                                         int BH, int hd, int n_split) {
  const int bh = blockIdx.x;
  const float* rec = scratch + (int64_t)bh * n_split * (hd + 2);
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, rec[s * (hd + 2)]);
  float L = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float ms = rec[s * (hd + 2)];
    if (ms != -INFINITY) L += __expf(ms - M) * rec[s * (hd + 2) + 1];
  }
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float ms = rec[s * (hd + 2)];
      if (ms != -INFINITY) a += __expf(ms - M) * rec[s * (hd + 2) + 2 + i];
    }
    o[(int64_t)bh * hd + i] = from_f32<T>(a / L);
  }
}

// ------------------------------------------------------------------- argmax
// One block per row; ties resolve to the lowest index (NaNs never win).
__global__ void argmax_kernel(const float* __restrict__ x, int n, int32_t* __restrict__ out) {
  const float* xr = x + (int64_t)blockIdx.x * n;
  float best = -INFINITY;
  int idx = n;  // sentinel larger than any index
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float v = xr[j];
    if (v > best || (v == best && j < idx)) {
      best = v;
      idx = j;
    }
  }
  __shared__ float sb[32];
  __shared__ int si[32];
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ob > best || (ob == best && oi < idx)) {
      best = ob;
      idx = oi;
    }
  }
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  if (lane == 0) {
    sb[wid] = best;
    si[wid] = idx;
  }
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x / 32;
    best = lane < nw ? sb[lane] : -INFINITY;
    idx = lane < nw ? si[lane] : n;
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ob > best || (ob == best && oi < idx)) {
        best = ob;
        idx = oi;
      }
    }
    if (lane == 0) out[blockIdx.x] = idx < n ? idx : 0;
  }
}

// y[b, :] = x[b*T + T-1, :]
__global__ void gather_last_rows_kernel(const float* __restrict__ x, float* __restrict__ y, int T,
                                        int d) {
  const int b = blockIdx.x;
  const float* src = x + ((int64_t)b * T + T - 1) * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) y[(int64_t)b * d + j] = src[j];
}

// ---------------------------------------------------------------- launchers
static inline unsigned grid_rows(int64_t rows, int per_block) {
  return (unsigned)((rows + per_block - 1) / per_block);
}

// Calls F<T>() with T the C++ type of an nc_dtype.
#define NC_DISPATCH(dt, T, ...)            \
  do {                                     \
    if ((dt) == NC_BF16) {                 \
      typedef bf16 T;                      \
      __VA_ARGS__;                         \
    } else if ((dt) == NC_F16) {           \
      typedef f16 T;                       \
      __VA_ARGS__;                         \
    } else {                               \
      typedef float T;                     \
      __VA_ARGS__;                         \
    }                                      \
  } while (0)

void launch_embed_norm(const int32_t* tok, const void* wte, nc_dtype wdt, float* x, void* xn,
                       nc_dtype adt, int64_t M, int d, int vocab, float eps, uint32_t* status,
                       cudaStream_t s) {
  count_launches(1);
  NC_DISPATCH(wdt, TW, NC_DISPATCH(adt, TA, (embed_norm_kernel<TW, TA><<<grid_rows(M, 8), 256, 0, s>>>(
                                              tok, (const TW*)wte, x, (TA*)xn, M, d, vocab, eps, status))));
}

void launch_rmsnorm(const float* x, void* y, nc_dtype ydt, int64_t M, int d, float eps,
                    cudaStream_t s) {
  count_launches(1);
  NC_DISPATCH(ydt, T, (rmsnorm_kernel<T><<<grid_rows(M, 8), 256, 0, s>>>(x, (T*)y, M, d, eps)));
}

void launch_gemm_simt(const void* A, const void* B, float* C, int64_t M, int N, int K,
                      int64_t ldc, nc_dtype dt, cudaStream_t s) {
  count_launches(1);
  dim3 grid((N + 63) / 64, (unsigned)((M + 63) / 64));
  NC_DISPATCH(dt, T, (gemm_simt_kernel<T><<<grid, 256, 0, s>>>((const T*)A, (const T*)B, C, M, N, K, ldc)));
}

void launch_qkv_post(const float* part, int n_split, int64_t M, const RowMap& rm,
                     const QkvDst& dst, nc_dtype dt, cudaStream_t s) {
  count_launches(1);
  const int64_t warps = M * (dst.H + 2 * dst.Hkv);
  NC_DISPATCH(dt, T, (qkv_post_kernel<T><<<grid_rows(warps, 8), 256, 0, s>>>(part, n_split, M, rm, dst)));
}

void launch_residual_finish(const float* part, int n_split, float* x, int64_t M, int N,
                            void* xn_out, nc_dtype dt, float eps, cudaStream_t s) {
  count_launches(1);
  NC_DISPATCH(dt, T, (residual_finish_kernel<T><<<grid_rows(M, 8), 256, 0, s>>>(part, n_split, x, M, N,
                                                                             (T*)xn_out, eps)));
}

void launch_relu2_finish(const float* part, int n_split, void* h, int64_t M, int N, nc_dtype dt,
                         uint32_t* status, cudaStream_t s) {
  count_launches(1);
  const int64_t total = M * N;
  const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, 148 * 16);
  NC_DISPATCH(dt, T, (relu2_finish_kernel<T><<<grid, 256, 0, s>>>(part, n_split, (T*)h, total, status)));
}

void launch_sum_splits(const float* part, int n_split, float* out, int64_t M, int N, int64_t ldo,
                       cudaStream_t s) {
  count_launches(1);
  const int64_t total = M * N;
  const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, 148 * 16);
  sum_splits_kernel<<<grid, 256, 0, s>>>(part, n_split, out, M, N, ldo);
}

void launch_attention_prefill_simt(const void* q, const void* k, const void* v, void* o, int B,
                                   int H, int Hkv, int T_, int t_max, int hd, nc_dtype dt,
                                   cudaStream_t s) {
  count_launches(1);
  const int64_t warps = (int64_t)B * H * T_;
  const size_t smem = 8 * hd * sizeof(float);
  NC_DISPATCH(dt, T, (attention_prefill_simt_kernel<T><<<grid_rows(warps, 8), 256, smem, s>>>(
                         (const T*)q, (const T*)k, (const T*)v, (T*)o, B, H, Hkv, T_, t_max, hd)));
}

void launch_attention_decode_simt(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int len, int t_max, int hd, nc_dtype dt,
                                  float* scratch, int n_split, cudaStream_t s) {
  count_launches(1);
  dim3 grid(B * H, n_split);
  const size_t smem = hd * sizeof(float);
  NC_DISPATCH(dt, T, (attention_decode_simt_kernel<T><<<grid, 32, smem, s>>>(
                          (const T*)q, (const T*)k, (const T*)v, scratch, B, H, Hkv, len, t_max, hd,
                          n_split)));
  launch_attention_combine(scratch, o, B * H, hd, n_split, dt, s);
}

void launch_attention_combine(const float* scratch, void* o, int BH, int hd, int n_split,
                              nc_dtype dt, cudaStream_t s) {
  count_launches(1);
  NC_DISPATCH(dt, T, (attention_combine_kernel<T><<<BH, 128, 0, s>>>(scratch, (T*)o, BH, hd,
                                                                     n_split)));
}

size_t decode_attention_scratch_bytes(int B, int H, int Hkv, int len, int hd) {
  int tps = 1, ns = 1;
  decode_attention_plan(len, B * Hkv, &tps, &ns);
  return (size_t)B * H * ns * (hd + 2) * sizeof(float);
}

void launch_attention_decode(const void* q, const void* k, const void* v, void* o, int B, int H,
                             int Hkv, int len, int t_max, int hd, nc_dtype dt, float* scratch,
                             cudaStream_t s) {
  if (decode_attention_mma_ok(H, Hkv, hd, dt)) {
    launch_attention_decode_mma(q, k, v, o, B, H, Hkv, len, t_max, dt, scratch, s);
    return;
  }
  int tps = 1, ns = 1;
  decode_attention_plan(len, B * Hkv, &tps, &ns);
  launch_attention_decode_simt(q, k, v, o, B, H, Hkv, len, t_max, hd, dt, scratch, ns, s);
}

void launch_argmax(const float* x, int rows, int n, int32_t* out, cudaStream_t s) {
  count_launches(1);
  argmax_kernel<<<rows, 1024, 0, s>>>(x, n, out);
}

void launch_gather_rows(const float* x, float* y, int B, int T, int d, cudaStream_t s) {
  count_launches(1);
  gather_last_rows_kernel<<<B, 256, 0, s>>>(x, y, T, d);
}

template <class TI, class TO>
__global__ void convert_kernel(const TI* __restrict__ src, TO* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f32<TO>(to_f32(src[i]));
}

void launch_convert16(const void* src, nc_dtype from, void* dst, nc_dtype to, int64_t n,
                      cudaStream_t s) {
  count_launches(1);
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 148 * 32);
  NC_DISPATCH(from, TI, NC_DISPATCH(to, TO, (convert_kernel<TI, TO><<<grid, 256, 0, s>>>(
                                                 (const TI*)src, (TO*)dst, n))));
}

}  // namespace nc
