// Causal flash attention for prefill (bf16, head_dim 128) with online fp32
// softmax and grouped-query head sharing.
//
// CTA = 4 warps = 64 query rows of one (sequence, query head); each warp owns 16
// rows. Key/value tiles of 64 positions stream through shared memory
// (cp.async, double buffered, 16-byte chunks XOR-swizzled by row). Scores
// S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate);
// the S fragments are reused in registers as the P operand. Query tiles are
// scheduled heaviest-first (the causal triangle makes late tiles longest).
#include <math.h>

#include "common.cuh"
#include "tc.h"

namespace nc {
namespace {

constexpr int kHd = 128;
constexpr int kBq = 64;        // query rows per CTA
constexpr int kBk = 64;        // key rows per tile
constexpr int kRowBytes = kHd * 2;   // 256
constexpr int kTileBytes = kBk * kRowBytes;  // 16 KB

// byte offset of 16-byte chunk c (0..15) of row r in a swizzled 256-byte-row tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
template <class T16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<bf16>(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<f16>(float (&c)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Loads rows [row0, row0 + 64) of a [rows, 128] bf16 matrix into a swizzled
// tile; rows >= row_limit are zero-filled.
template <class T16>
__device__ __forceinline__ void load_tile(uint32_t dst, const T16* src, int row0, int row_limit) {
  for (int i = threadIdx.x; i < kBk * 16; i += 128) {
    const int r = i / 16, c = i % 16;
    const bool ok = row0 + r < row_limit;
    const T16* p = src + (int64_t)(ok ? row0 + r : 0) * kHd + c * 8;
    cp_async16(dst + swz(r, c), p, ok);
  }
}

template <class T16>
__global__ void __launch_bounds__(128) attn_prefill_mma_kernel(const T16* __restrict__ q,
                                                               const T16* __restrict__ k,
                                                               const T16* __restrict__ v,
                                                               T16* __restrict__ o, int H, int Hkv,
                                                               int T, int t_max, float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + kTileBytes;   // K[2], then V[2]
  const int num_qt = (T + kBq - 1) / kBq;
  const int qt = num_qt - 1 - (int)blockIdx.x;   // heaviest first
  const int bh = blockIdx.y;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / Hkv);
  const int q0 = qt * kBq;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const T16* qb = q + ((int64_t)b * H + h) * T * kHd;
  const T16* kb = k + ((int64_t)b * Hkv + g) * t_max * kHd;
  const T16* vb = v + ((int64_t)b * Hkv + g) * t_max * kHd;

  const int n_kv = qt + 1;   // causal: key tiles 0..qt
  load_tile(sQ, qb, q0, T);
  load_tile(sK0, kb, 0, T);
  load_tile(sK0 + 2 * kTileBytes, vb, 0, T);
  cp_async_commit();

  float oacc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  uint32_t qf[8][4];
  const int gq = lane / 4, tq = lane % 4;

  for (int j = 0; j < n_kv; ++j) {
    const int buf = j & 1;
    if (j + 1 < n_kv) {
      load_tile(sK0 + (buf ^ 1) * kTileBytes, kb, (j + 1) * kBk, T);
      load_tile(sK0 + (2 + (buf ^ 1)) * kTileBytes, vb, (j + 1) * kBk, T);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
      // Q fragments of this warp's 16 rows, all 8 k-steps of the head dim
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int r = warp * 16 + (lane % 16);
        const int c = ks * 2 + lane / 16;
        ldsm_x4(sQ + swz(r, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const uint32_t sK = sK0 + buf * kTileBytes;
    const uint32_t sV = sK0 + (2 + buf) * kTileBytes;
    // S = Q K^T for 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int r = np * 16 + (lane / 16) * 8 + (lane % 8);
        const int c = ks * 2 + (lane / 8) % 2;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + swz(r, c), b0, b1, b2, b3);
        mma16816<T16>(s[2 * np], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
        mma16816<T16>(s[2 * np + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
      }
    }
    // causal mask on the diagonal tile
    if (j == qt) {
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = q0 + warp * 16 + gq + (e / 2) * 8;
          const int key = j * kBk + n * 8 + 2 * tq + (e % 2);
          if (key > row) s[n][e] = -INFINITY;
        }
    }
    // online softmax (rows gq and gq + 8 of the warp)
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2], rs[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) corr[r] = exp2f((m_run[r] - mx[r]) * scale_log2);
    uint32_t pf[8][2];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2f((s[n][0] - mx[0]) * scale_log2);
      const float p1 = exp2f((s[n][1] - mx[0]) * scale_log2);
      const float p2 = exp2f((s[n][2] - mx[1]) * scale_log2);
      const float p3 = exp2f((s[n][3] - mx[1]) * scale_log2);
      rs[0] += p0 + p1;
      rs[1] += p2 + p3;
      pf[n][0] = pack2<T16>(p0, p1);
      pf[n][1] = pack2<T16>(p2, p3);
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
      oacc[i][0] *= corr[0];
      oacc[i][1] *= corr[0];
      oacc[i][2] *= corr[1];
      oacc[i][3] *= corr[1];
    }
    // O += P V : k = 64 keys (4 steps of 16), n = 128 dims (16 tiles of 8)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t a0 = pf[2 * kk][0], a1 = pf[2 * kk][1], a2 = pf[2 * kk + 1][0],
                     a3 = pf[2 * kk + 1][1];
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int r = kk * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
        const int c = dp * 2 + lane / 16;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV + swz(r, c), b0, b1, b2, b3);
        mma16816<T16>(oacc[2 * dp], a0, a1, a2, a3, b0, b1);
        mma16816<T16>(oacc[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }
  // normalise and store o[b][t][h*128 + dim]
  const float inv[2] = {1.f / l_run[0], 1.f / l_run[1]};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = q0 + warp * 16 + gq + r * 8;
    if (t >= T) continue;
    T16* out = o + ((int64_t)b * T + t) * H * kHd + (int64_t)h * kHd;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int dim = i * 8 + 2 * tq;
      *reinterpret_cast<uint32_t*>(out + dim) =
          pack2<T16>(oacc[i][2 * r] * inv[r], oacc[i][2 * r + 1] * inv[r]);
    }
  }
}

template <class T16>
nc_status launch_attn(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv,
                      int T, int t_max, cudaStream_t s) {
  const size_t smem = 5 * kTileBytes;
  if (!ensure_dyn_smem((const void*)attn_prefill_mma_kernel<T16>, smem)) return NC_ERR_CUDA;
  dim3 grid((T + kBq - 1) / kBq, B * H);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kHd);
  attn_prefill_mma_kernel<T16><<<grid, 128, smem, s>>>((const T16*)q, (const T16*)k,
                                                       (const T16*)v, (T16*)o, H, Hkv, T, t_max,
                                                       scale_log2);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace

nc_status tc_attention_prefill(const void* q, const void* k, const void* v, void* o, int B, int H,
                               int Hkv, int T, int t_max, nc_dtype dt, cudaStream_t s) {
  if (dt == NC_F16) return launch_attn<f16>(q, k, v, o, B, H, Hkv, T, t_max, s);
  return launch_attn<bf16>(q, k, v, o, B, H, Hkv, T, t_max, s);
}

}  // namespace nc
