// Decode attention on tensor cores: one query position per sequence against the
// KV cache, split over key ranges, for head_dim 128 and up to 16 query heads per
// KV head.
//
// CTA (4 warps) = one (sequence b, KV head g, key range). The G query heads that
// share KV head g form the 16-row A operand of mma.sync m16n8k16 (rows >= G are
// zero), so one pass over K/V serves the whole group -- with MQA (G = 10) the
// cache is read once for ten heads. Key tiles of 64 positions stream through
// shared memory with cp.async (double buffered); warp w takes keys [16w, 16w+16)
// of each tile and keeps its own online-softmax state; the four states are merged
// in shared memory and the CTA writes one partial (m, l, o) per query head, in the
// layout the log-sum-exp combine kernel reads.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

constexpr int kHd = 128;
constexpr int kTile = 64;
constexpr int kRowBytes = kHd * 2;
constexpr int kTileBytes = kTile * kRowBytes;   // 16 KB
constexpr int kQBytes = 16 * kRowBytes;         // 4 KB

__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
template <class T16>
__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma<f16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma<bf16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// rows [row0, row0 + 64) of a [rows, 128] matrix into a swizzled tile; rows >= limit -> 0
template <class T16>
__device__ __forceinline__ void load_tile(uint32_t dst, const T16* src, int row0, int limit) {
  for (int i = threadIdx.x; i < kTile * 16; i += 128) {
    const int r = i / 16, c = i % 16;
    const bool ok = row0 + r < limit;
    cp_async16(dst + swz(r, c), src + (int64_t)(ok ? row0 + r : 0) * kHd + c * 8, ok);
  }
}

template <class T16>
__global__ void __launch_bounds__(128) attn_decode_mma_kernel(
    const T16* __restrict__ q, const T16* __restrict__ k, const T16* __restrict__ v,
    float* __restrict__ scratch, int H, int Hkv, int len, int t_max, int n_split,
    int tiles_per_split, float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + kQBytes;   // K[2] then V[2]
  const int split = blockIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int G = H / Hkv;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int gq = lane / 4, tq = lane % 4;
  const int k0 = split * tiles_per_split * kTile;
  const int k1 = min(len, k0 + tiles_per_split * kTile);
  const float ln2 = 0.6931471805599453f;

  if (k0 >= k1) {   // empty range: neutral partial state
    for (int r = warp; r < G; r += 4) {
      float* rec = scratch + (((int64_t)b * H + g * G + r) * n_split + split) * (kHd + 2);
      for (int i = lane; i < kHd + 2; i += 32) rec[i] = i == 0 ? -INFINITY : 0.f;
    }
    return;
  }
  // Q rows of the group (rows >= G zero-filled)
  const T16* qg = q + ((int64_t)b * H + g * G) * kHd;
  for (int i = threadIdx.x; i < 16 * 16; i += 128) {
    const int r = i / 16, c = i % 16;
    const bool ok = r < G;
    cp_async16(sQ + swz(r, c), qg + (int64_t)(ok ? r : 0) * kHd + c * 8, ok);
  }
  const T16* kb = k + (int64_t)bg * t_max * kHd;
  const T16* vb = v + (int64_t)bg * t_max * kHd;
  const int n_t = (k1 - k0 + kTile - 1) / kTile;
  load_tile(sKV, kb, k0, k1);
  load_tile(sKV + 2 * kTileBytes, vb, k0, k1);
  cp_async_commit();

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  uint32_t qf[8][4];

  for (int j = 0; j < n_t; ++j) {
    const int buf = j & 1;
    if (j + 1 < n_t) {
      load_tile(sKV + (buf ^ 1) * kTileBytes, kb, k0 + (j + 1) * kTile, k1);
      load_tile(sKV + (2 + (buf ^ 1)) * kTileBytes, vb, k0 + (j + 1) * kTile, k1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        ldsm_x4(sQ + swz(lane % 16, ks * 2 + lane / 16), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
    const uint32_t sK = sKV + buf * kTileBytes, sV = sKV + (2 + buf) * kTileBytes;
    // scores of this warp's 16 keys: two n-tiles of 8
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sK + swz(warp * 16 + (lane / 16) * 8 + (lane % 8), ks * 2 + (lane / 8) % 2), b0, b1,
              b2, b3);
      mma<T16>(s[0], qf[ks], b0, b1);
      mma<T16>(s[1], qf[ks], b2, b3);
    }
    const int kbase = k0 + j * kTile + warp * 16;
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (kbase + n * 8 + 2 * tq + (e % 2) >= k1) s[n][e] = -INFINITY;
        mx[e / 2] = fmaxf(mx[e / 2], s[n][e]);
      }
    float corr[2], rs[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      corr[r] = mx[r] == -INFINITY ? 1.f : ex2_approx((m_run[r] - mx[r]) * scale_log2);
    }
    uint32_t a[4];
    {
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = mx[e / 2];
          p[n][e] = m == -INFINITY ? 0.f : ex2_approx((s[n][e] - m) * scale_log2);
          rs[e / 2] += p[n][e];
        }
      a[0] = pack2<T16>(p[0][0], p[0][1]);
      a[1] = pack2<T16>(p[0][2], p[0][3]);
      a[2] = pack2<T16>(p[1][0], p[1][1]);
      a[3] = pack2<T16>(p[1][2], p[1][3]);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
      l_run[r] = l_run[r] * corr[r] + rs[r];
      m_run[r] = mx[r];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= corr[0];
      o[i][1] *= corr[0];
      o[i][2] *= corr[1];
      o[i][3] *= corr[1];
    }
    // O += P V over this warp's 16 keys (one k-step), 16 dim tiles
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sV + swz(warp * 16 + (lane % 8) + ((lane / 8) % 2) * 8, dp * 2 + lane / 16), b0, b1,
                b2, b3);
      mma<T16>(o[2 * dp], a, b0, b1);
      mma<T16>(o[2 * dp + 1], a, b2, b3);
    }
    __syncthreads();
  }

  // merge the four warps' states: M = max_w m_w, weights e^(m_w - M)
  float* red = reinterpret_cast<float*>(smem + kQBytes);   // reuses the K/V buffers
  float* wm = red;                 // [4][16]
  float* wl = red + 64;            // [4][16]
  float* wo = red + 128;           // [4][16][128]
  if (tq == 0) {
    wm[warp * 16 + gq] = m_run[0];
    wm[warp * 16 + gq + 8] = m_run[1];
    wl[warp * 16 + gq] = l_run[0];
    wl[warp * 16 + gq + 8] = l_run[1];
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int dim = i * 8 + 2 * tq;
    wo[(warp * 16 + gq) * kHd + dim] = o[i][0];
    wo[(warp * 16 + gq) * kHd + dim + 1] = o[i][1];
    wo[(warp * 16 + gq + 8) * kHd + dim] = o[i][2];
    wo[(warp * 16 + gq + 8) * kHd + dim + 1] = o[i][3];
  }
  __syncthreads();
  for (int r = warp; r < G; r += 4) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * 16 + r]);
    float sc[4], L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      sc[w] = wm[w * 16 + r] == -INFINITY ? 0.f : ex2_approx((wm[w * 16 + r] - M) * scale_log2);
      L += sc[w] * wl[w * 16 + r];
    }
    float* rec = scratch + (((int64_t)b * H + g * G + r) * n_split + split) * (kHd + 2);
    if (lane == 0) {
      rec[0] = M * scale_log2 * ln2;   // natural-log units, as the combine kernel expects
      rec[1] = L;
    }
    for (int i = lane; i < kHd; i += 32) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) acc += sc[w] * wo[(w * 16 + r) * kHd + i];
      rec[2 + i] = acc;
    }
  }
}

}  // namespace

void decode_attention_plan(int len, int bg, int* tiles_per_split, int* n_split) {
  const int tiles = (len + kTile - 1) / kTile;
  const int want = std::max(1, 296 / std::max(1, bg));   // about two CTAs per SM
  int tps = (tiles + want - 1) / want;
  tps = std::max(tps, (tiles + 63) / 64);                 // at most 64 splits
  tps = std::max(1, tps);
  *tiles_per_split = tps;
  *n_split = (tiles + tps - 1) / tps;
}

bool decode_attention_mma_ok(int H, int Hkv, int hd, nc_dtype dt) {
  return hd == kHd && H / Hkv <= 16 && (dt == NC_F16 || dt == NC_BF16);
}

void launch_attention_decode_mma(const void* q, const void* k, const void* v, void* o, int B,
                                 int H, int Hkv, int len, int t_max, nc_dtype dt, float* scratch,
                                 cudaStream_t s) {
  int tps = 1, ns = 1;
  decode_attention_plan(len, B * Hkv, &tps, &ns);
  const size_t smem = kQBytes + 4 * kTileBytes;   // >= the merge area (4*16*130 floats)
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kHd);
  dim3 grid(ns, B * Hkv);
  if (dt == NC_F16) {
    // a refusal leaves the launch below to fail, which the caller's error check reports
    ensure_dyn_smem((const void*)attn_decode_mma_kernel<f16>, smem);
    attn_decode_mma_kernel<f16><<<grid, 128, smem, s>>>((const f16*)q, (const f16*)k, (const f16*)v,
                                                         scratch, H, Hkv, len, t_max, ns, tps,
                                                         scale_log2);
  } else {
    ensure_dyn_smem((const void*)attn_decode_mma_kernel<bf16>, smem);
    attn_decode_mma_kernel<bf16><<<grid, 128, smem, s>>>((const bf16*)q, (const bf16*)k,
                                                          (const bf16*)v, scratch, H, Hkv, len,
                                                          t_max, ns, tps, scale_log2);
  }
  count_launches(1);
  launch_attention_combine(scratch, o, B * H, kHd, ns, dt, s);
}

}  // namespace nc
