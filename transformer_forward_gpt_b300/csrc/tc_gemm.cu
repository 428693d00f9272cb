// tcgen05 GEMM for sm_103a: C = A B^T with bf16 operands staged by TMA into
// shared memory (128-byte swizzle, K-major), fp32 accumulators in TMEM, and the
// epilogue read back with tcgen05.ld.
//
// Persistent, warp-specialised CTA of 192 threads:
//   warp 0      one thread issues the TMA loads of A and B into a ring of stages
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (128 x BN x 16) and
//               commits to mbarriers that free a stage / publish an accumulator
//   warps 2..5  epilogue: warp w reads TMEM lanes 32*(w%4)..+31, so each thread
//               owns one output row of the 128-row tile
// Two TMEM accumulators (2*BN columns) let the epilogue of one tile overlap the
// main loop of the next.
//
// Two ways the projections of the forward pass are laid onto it:
//   tile mode (many token rows): A = activations [M, K], B = weights [N, K]; the
//     epilogue is fused: RoPE + QK norm + scatter (Q/K/V), residual add (O, PROJ),
//     ReLU^2 (FC) or an fp32 store (LM head).
//   swap mode (<= 128 token rows, decode): A = weights, B = activations, so the
//     weights fill the 128-row MMA; K may be split across CTAs. The epilogue
//     writes transposed fp32 partial sums [split][token][feature] that a
//     finishing kernel reduces (or, unsplit, the logits directly).
#include <limits.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "tc.h"

namespace nc {

enum Epi : int { EPI_F32 = 0, EPI_RESID = 1, EPI_RELU2 = 2, EPI_QKV = 3, EPI_SWAP = 4, EPI_CE = 5 };

struct GemmArgs {
  int M;                  // rows of the A operand
  int N;                  // rows of the B operand
  int num_m_blk, num_n_blk, num_k_blk;
  int k_splits, k_per_split;
  int a_split0, a_split1;  // row boundaries between A tensor maps 0 | 1 | 2
  int b_split0, b_split1;  // the same for B (multiples of 128)
  float* out_f32;          // EPI_F32 (C), EPI_RESID (x), EPI_SWAP (partials or logits)
  void* out_16;            // EPI_RELU2 (16-bit type of the kernel)
  int64_t ldo;             // row pitch of the output, elements
  int64_t split_stride;    // EPI_SWAP: elements between split slices
  RowMap rm;               // EPI_QKV
  QkvDst qkv;
  uint32_t* status;
  int stream_k;            // 1: CTAs take equal contiguous ranges of (tile, k block)
  int sk_groups;           // > 1 (stream-K): one group of CTAs per n block, see Sched
  const float* row_scale;  // EPI_SWAP with 8-bit operands: scale of each A row (feature)
  const float* tok_scale;  // and of each B row (token); NULL for 16-bit operands
  const int32_t* targets;  // EPI_CE: target column of each row (out_f32: float2 partials)
  float* ce_zt;            // EPI_CE: the target column's value of each row
  int c_tma;               // EPI_F32, EPI_RELU2: store the output through tmC by TMA
};

// Work schedule shared by the three roles of a CTA: a sequence of segments
// (m block, n block, k blocks [kb0, kb1), split index for EPI_SWAP).
//   persistent: whole tiles (or K splits) u = first, first + step, ...
//   stream-K:   the CTA's contiguous share of all (tile, k block) pairs, so
//               every CTA does the same number of k blocks; a tile cut between
//               CTAs is finished by more than one of them (EPI_RESID adds).
//               Tiles are ordered n block fastest.
//   grouped stream-K (sk_groups = n blocks = G): CTA c works on n block c % G
//               and takes share c / G of the (m block, k block) pairs, the same
//               share in every group; the G CTAs that need one k block of A then
//               read it at about the same time, so L2 serves it to all but the
//               first. CTAs past the last full group of G stay idle.
struct Seg {
  int mb, nb, kb0, kb1, ks;
};
struct Sched {
  int64_t pos, end;   // stream-K position / end, or persistent unit / units
  int step;
  int nbf;            // grouped stream-K: this CTA's n block (else -1)
  bool sk;
  __device__ __forceinline__ void init(const GemmArgs& p) {
    sk = p.stream_k != 0;
    nbf = -1;
    if (sk && p.sk_groups > 1) {
      const int G = p.sk_groups, P = (int)gridDim.x / G, c = (int)blockIdx.x;
      const int64_t total = (int64_t)p.num_m_blk * p.num_k_blk;
      nbf = c % G;
      pos = c < G * P ? total * (c / G) / P : 0;
      end = c < G * P ? total * (c / G + 1) / P : 0;
      step = 0;
    } else if (sk) {
      const int64_t total = (int64_t)p.num_m_blk * p.num_n_blk * p.num_k_blk;
      pos = total * blockIdx.x / gridDim.x;
      end = total * (blockIdx.x + 1) / gridDim.x;
      step = 0;
    } else {
      pos = blockIdx.x;
      end = (int64_t)p.num_m_blk * p.num_n_blk * p.k_splits;
      step = gridDim.x;
    }
  }
  __device__ __forceinline__ bool next(const GemmArgs& p, Seg& g) {
    if (pos >= end) return false;
    if (sk && nbf >= 0) {
      g.kb0 = (int)(pos % p.num_k_blk);
      { const int64_t e = g.kb0 + (end - pos); g.kb1 = (int)(e < p.num_k_blk ? e : p.num_k_blk); }
      g.nb = nbf;
      g.mb = (int)(pos / p.num_k_blk);
      g.ks = 0;
      pos += g.kb1 - g.kb0;
    } else if (sk) {
      // tiles n-block fastest: the n tiles of one 128-row block of A follow one
      // another, so that block is read from DRAM once and from L2 after (A of
      // the PROJ projection, 84 MB at d20, does not stay in L2 across a sweep)
      const int64_t t = pos / p.num_k_blk;
      g.kb0 = (int)(pos % p.num_k_blk);
      { const int64_t e = g.kb0 + (end - pos); g.kb1 = (int)(e < p.num_k_blk ? e : p.num_k_blk); }
      g.nb = (int)(t % p.num_n_blk);
      g.mb = (int)(t / p.num_n_blk);
      g.ks = 0;
      pos += g.kb1 - g.kb0;
    } else {
      const int u = (int)pos;
      g.mb = u % p.num_m_blk;
      const int rest = u / p.num_m_blk;
      g.nb = rest % p.num_n_blk;
      g.ks = rest / p.num_n_blk;
      g.kb0 = g.ks * p.k_per_split;
      g.kb1 = min(p.num_k_blk, g.kb0 + p.k_per_split);
      pos += step;
    }
    return true;
  }
};

template <int BN>
struct TileCfg {
  static constexpr int kABytes = 128 * 64 * 2;
  static constexpr int kBBytes = BN * 64 * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (196608 / kStageBytes) > 8 ? 8 : (196608 / kStageBytes);
  static constexpr int kBoxRowsB = BN < 128 ? BN : 128;
  static constexpr int kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
  static constexpr int kEpiStride = 36;   // floats per staged row (16-byte aligned, conflict-free)
  static constexpr int kEpiBytes = 4 * 32 * kEpiStride * 4;
  static constexpr int kEpiTmaBytes = 4 * 32 * 128;   // per warp 32 rows x 128 B, swizzled
  // stages | barriers (1 KB) | epilogue staging (1024-aligned) ; + 1 KB of alignment slack
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 + 1024 +
                                       (kEpiBytes > kEpiTmaBytes ? kEpiBytes : kEpiTmaBytes);
};

__device__ __forceinline__ const CUtensorMap* pick_map(const CUtensorMap* m0, const CUtensorMap* m1,
                                                       const CUtensorMap* m2, int row, int s0,
                                                       int s1, int& local) {
  if (row < s0) {
    local = row;
    return m0;
  }
  if (row < s1) {
    local = row - s0;
    return m1;
  }
  local = row - s1;
  return m2;
}

// ----------------------------------------------------------------- epilogues
// Each thread holds row `row` of the tile; taddr points at its TMEM lane and
// the accumulator's first column. tcgen05.ld is warp-collective, so every lane
// runs the loads. A thread-per-row store would touch 32 rows per warp
// instruction, so each 32-column chunk goes through the warp's staging area
// (32 rows x kEpiStride floats) and is written row by row: 8 lanes cover the
// 128 bytes of one fp32 row chunk (4 lanes the 64 bytes of a 16-bit one).
template <int BN, class T16>
__device__ __forceinline__ void epi_store_rows(const GemmArgs& p, uint32_t taddr, float* stage,
                                               int row0, int nb, int mode) {
  constexpr int S = TileCfg<BN>::kEpiStride;
  const int lane = threadIdx.x % 32;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32_sync(taddr + c * 32, v);
    const int n0 = nb * BN + c * 32;
    if (n0 >= p.N) continue;   // uniform across the warp
    if (mode == EPI_RELU2) {
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float r = fmaxf(v[j], 0.f);
        v[j] = r * r;
        amax = fmaxf(amax, v[j]);
      }
      note_range<T16>(amax, p.status);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(stage + lane * S + 4 * i) =
          make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    __syncwarp();
    if (mode == EPI_RELU2) {
      // 4 lanes per row (8 values each), 8 rows per pass
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int r = it * 8 + lane / 4, cc = (lane % 4) * 8;
        const int grow = row0 + r, gcol = n0 + cc;
        if (grow < p.M && gcol < p.N) {
          const float4 a = *reinterpret_cast<const float4*>(stage + r * S + cc);
          const float4 b = *reinterpret_cast<const float4*>(stage + r * S + cc + 4);
          T16* dst = reinterpret_cast<T16*>(p.out_16) + (int64_t)grow * p.ldo + gcol;
          *reinterpret_cast<uint4*>(dst) = make_uint4(pack2<T16>(a.x, a.y), pack2<T16>(a.z, a.w),
                                                      pack2<T16>(b.x, b.y), pack2<T16>(b.z, b.w));
        }
      }
    } else {
      // 8 lanes per row (4 values each), 4 rows per pass. The residual add is a
      // vector reduction into x: no load, and a tile split between CTAs
      // (stream-K) adds each part.
      const int cc = (lane % 8) * 4, gcol = n0 + cc;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int r = it * 4 + lane / 8;
        const int grow = row0 + r;
        if (grow < p.M && gcol < p.N) {
          const float4 a = *reinterpret_cast<const float4*>(stage + r * S + cc);
          float* dst = p.out_f32 + (int64_t)grow * p.ldo + gcol;
          if (mode == EPI_RESID) {
            red_add_f32x4(dst, a);
          } else {
            st_global_cs_v4(dst, make_uint4(__float_as_uint(a.x), __float_as_uint(a.y),
                                            __float_as_uint(a.z), __float_as_uint(a.w)));
          }
        }
      }
    }
    __syncwarp();
  }
}

// Q/K/V epilogue: the tile's BN columns are BN/128 whole heads of the
// concatenated [Q | K | V] projection. For Q and K heads: the mean square is
// taken over the un-rotated values (the rotation keeps the norm), then pairs
// (i, i + 64) are rotated by +theta(t, i) and scaled by the QK-norm factor.
template <int BN, class T16>
__device__ __forceinline__ void epi_qkv(const GemmArgs& p, uint32_t taddr, int row, int nb) {
  const QkvDst& q = p.qkv;
  const bool valid = row < p.M;
  const int total_heads = q.H + 2 * q.Hkv;
  const int b = valid ? row / p.rm.rows_per_seq : 0;
  const int t = valid ? p.rm.pos0 + row % p.rm.rows_per_seq : 0;
#pragma unroll 1
  for (int hc = 0; hc < BN / 128; ++hc) {
    const int j = nb * (BN / 128) + hc;
    if (j >= total_heads) break;
    const uint32_t base = taddr + hc * 128;
    if (j >= q.H + q.Hkv) {  // V head, stored as projected
      const int g = j - q.H - q.Hkv;
      T16* out = reinterpret_cast<T16*>(q.v_cache) + (((int64_t)b * q.Hkv + g) * q.t_max + t) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32_sync(base + c * 32, v);
        if (valid) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
          note_range<T16>(amax, p.status);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(out + c * 32 + 8 * i) = make_uint4(
                pack2<T16>(v[8 * i], v[8 * i + 1]), pack2<T16>(v[8 * i + 2], v[8 * i + 3]),
                pack2<T16>(v[8 * i + 4], v[8 * i + 5]), pack2<T16>(v[8 * i + 6], v[8 * i + 7]));
        }
      }
      continue;
    }
    // the head's 128 values in one TMEM load; mean square over the un-rotated values
    float hv[128];
    tmem_ld128_sync(base, hv);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 128; ++i) ss = fmaf(hv[i], hv[i], ss);
    const float r = rsqrtf(ss * (1.f / 128.f) + q.eps);
    if (!valid) continue;
    T16* out;
    if (j < q.H)
      out = reinterpret_cast<T16*>(q.q) +
            (((int64_t)b * q.H + j) * p.rm.rows_per_seq + (t - p.rm.pos0)) * 128;
    else
      out = reinterpret_cast<T16*>(q.k_cache) + (((int64_t)b * q.Hkv + (j - q.H)) * q.t_max + t) * 128;
    // position-minor tables: entry i of position t at [i * ld + t], so the warp's
    // 32 consecutive positions read one line per entry
    const float* cs = q.cos_t + t;
    const float* sn = q.sin_t + t;
    const int64_t ld = q.tab_ld;
    // pairs (i, i + 64) in four blocks of 16, each rotated, scaled and stored at once
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float lo[16], hi[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float cc = __ldg(cs + (16 * c + u) * ld), sv = __ldg(sn + (16 * c + u) * ld);
        const float a = hv[16 * c + u], h = hv[64 + 16 * c + u];
        lo[u] = (a * cc - h * sv) * r;
        hi[u] = (a * sv + h * cc) * r;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        *reinterpret_cast<uint4*>(out + 16 * c + 8 * i) = make_uint4(
            pack2<T16>(lo[8 * i], lo[8 * i + 1]), pack2<T16>(lo[8 * i + 2], lo[8 * i + 3]),
            pack2<T16>(lo[8 * i + 4], lo[8 * i + 5]), pack2<T16>(lo[8 * i + 6], lo[8 * i + 7]));
        *reinterpret_cast<uint4*>(out + 64 + 16 * c + 8 * i) = make_uint4(
            pack2<T16>(hi[8 * i], hi[8 * i + 1]), pack2<T16>(hi[8 * i + 2], hi[8 * i + 3]),
            pack2<T16>(hi[8 * i + 4], hi[8 * i + 5]), pack2<T16>(hi[8 * i + 6], hi[8 * i + 7]));
      }
    }
  }
}

// Swap mode: the thread's row is a weight row (output feature f); TMEM columns
// are tokens. Writes out[ks][token][f] (lanes of a warp write consecutive f).
template <int BN>
__device__ __forceinline__ void epi_swap(const GemmArgs& p, uint32_t taddr, int f, int nb, int ks) {
  const bool valid = f < p.M;
  float* base = p.out_f32 + (int64_t)ks * p.split_stride + f;
  // 8-bit operands: the codes' product times the feature's and the token's scale
  const float rs = (p.row_scale && valid) ? p.row_scale[f] : 1.f;
#pragma unroll 1
  for (int c = 0; c < BN / 16; ++c) {
    float v[16];
    tmem_ld16_sync(taddr + c * 16, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = nb * BN + c * 16 + i;
      if (valid && tok < p.N) base[(int64_t)tok * p.ldo] = p.tok_scale ? v[i] * rs * p.tok_scale[tok] : v[i];
    }
  }
}

// fp32 store of the tile through TMA: per 32-column chunk the warp writes its 32
// rows x 128 bytes into a 1024-aligned staging area in the 128-byte swizzled
// layout of the tensor map (16-byte chunk j of row r at position j ^ (r % 8)),
// and one lane issues the bulk tensor store. The staging area is rewritten only
// after the previous store has read it. Rows past M are clipped by the copy; a
// slab that starts past M is skipped.
template <int BN>
__device__ __forceinline__ void epi_store_tma(const GemmArgs& p, const CUtensorMap* tmC,
                                              uint32_t taddr, uint8_t* stage, int row0, int nb) {
  const int lane = threadIdx.x % 32;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32_sync(taddr + c * 32, v);
    const int n0 = nb * BN + c * 32;
    if (n0 >= p.N || row0 >= p.M) continue;   // uniform across the warp
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, stage, n0, row0);
      bulk_commit();
    }
  }
}

// The same for the 16-bit ReLU^2 output: two 32-column chunks become one box of
// 64 values per row (128 bytes, the same swizzled layout).
template <int BN, class T16>
__device__ __forceinline__ void epi_store_tma_relu2(const GemmArgs& p, const CUtensorMap* tmC,
                                                    uint32_t taddr, uint8_t* stage, int row0,
                                                    int nb) {
  static_assert(BN % 64 == 0, "pairs of 32-column chunks");
  const int lane = threadIdx.x % 32;
#pragma unroll 1
  for (int c = 0; c < BN / 64; ++c) {
    uint32_t w[32];
    float amax = 0.f;
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      float v[32];
      tmem_ld32_sync(taddr + c * 64 + hlf * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float r = fmaxf(v[j], 0.f);
        v[j] = r * r;
        amax = fmaxf(amax, v[j]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) w[hlf * 16 + j] = pack2<T16>(v[2 * j], v[2 * j + 1]);
    }
    const int n0 = nb * BN + c * 64;
    if (n0 >= p.N || row0 >= p.M) continue;   // uniform across the warp
    if (row0 + lane < p.M) note_range<T16>(amax, p.status);
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) =
          make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, stage, n0, row0);
      bulk_commit();
    }
  }
}

// Cross-entropy epilogue: the thread's row of the tile's BN logits becomes the
// pair (m, s) = (max z, sum exp(z - m)) over the columns below N, stored at
// part[nb][row] (lanes of a warp write consecutive rows); the value of the
// row's target column goes to ce_zt[row]. No logit leaves the SM.
template <int BN>
__device__ __forceinline__ void epi_ce(const GemmArgs& p, uint32_t taddr, int row, int nb) {
  constexpr float kLog2e = 1.4426950408889634f;
  const bool valid = row < p.M;
  const int tgt = valid ? __ldg(p.targets + row) : -1;
  float m = -INFINITY, s = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32_sync(taddr + c * 32, v);
    const int n0 = nb * BN + c * 32;
    if (n0 >= p.N) continue;   // uniform across the warp
    const int nv = min(32, p.N - n0);
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) cm = fmaxf(cm, v[j]);
    if (cm > m) {
      s *= exp2f((m - cm) * kLog2e);   // 0 while m is -inf (s is 0 then)
      m = cm;
    }
    // exp(z - m) = 2^(z log2 e - m log2 e), four independent partial sums
    const float ml = m * kLog2e;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) s4[j & 3] += exp2f(fmaf(v[j], kLog2e, -ml));
    s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    if (tgt >= n0 && tgt < n0 + nv) {
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j == tgt) z = v[j];
      p.ce_zt[row] = z;
    }
  }
  if (valid)
    reinterpret_cast<float2*>(p.out_f32)[(int64_t)nb * p.M + row] = make_float2(m, s);
}

// --------------------------------------------------------------------- kernel
template <int BN, int EPI, class T16>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs p) {
  using C = TileCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;  // [2] accumulator drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_stage = reinterpret_cast<float*>(smem + S * C::kStageBytes + 1024);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      Sched sc;
      sc.init(p);
      Seg sg;
      while (!*abort_flag && sc.next(p, sg)) {
        const int mb = sg.mb, nb = sg.nb;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* sa = smem + stage * C::kStageBytes;
          uint8_t* sb = sa + C::kABytes;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          int local;
          const CUtensorMap* ma = pick_map(&tmA0, &tmA1, &tmA2, mb * 128, p.a_split0, p.a_split1, local);
          constexpr int kElemsPerRow = 128 / (int)sizeof(T16);   // one 128-byte swizzle row
          tma_load_2d(sa, ma, &full[stage], kb * kElemsPerRow, local);
#pragma unroll
          for (int h = 0; h < BN / C::kBoxRowsB; ++h) {
            const CUtensorMap* mb_ = pick_map(&tmB0, &tmB1, &tmB2, nb * BN + h * C::kBoxRowsB,
                                              p.b_split0, p.b_split1, local);
            tma_load_2d(sb + h * C::kBoxRowsB * 128, mb_, &full[stage], kb * kElemsPerRow, local);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
          ++issued;
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA's shared memory goes away
        for (int i = 1; i <= min(issued, S); ++i) {
          const int st = (stage - i + S) % S;
          const uint32_t ph = (stage - i < 0) ? (phase ^ 1) : phase;
          mbar_wait(&full[st], ph, p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_f32acc(Fmt16<T16>::code, 128, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      Sched sc;
      sc.init(p);
      Seg sg;
      while (!*abort_flag && sc.next(p, sg)) {
        const int kb0 = sg.kb0, kb1 = sg.kb1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.status)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_ss<T16>(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32),
                        sdesc_kmajor_sw128(b_addr + k * 32), kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp % 4;
    int acc = 0;
    uint32_t acc_phase = 0;
    Sched sc;
    sc.init(p);
    Seg sg;
    while (sc.next(p, sg)) {
      const int mb = sg.mb, nb = sg.nb, ks = sg.ks;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, p.status));
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      __syncwarp();
      tc_fence_after();
      const int row = mb * 128 + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if constexpr (EPI == EPI_SWAP)
        epi_swap<BN>(p, taddr, row, nb, ks);
      else if constexpr (EPI == EPI_QKV)
        epi_qkv<BN, T16>(p, taddr, row, nb);
      else if constexpr (EPI == EPI_CE)
        epi_ce<BN>(p, taddr, row, nb);
      else if (EPI == EPI_F32 && p.c_tma)
        epi_store_tma<BN>(p, &tmC, taddr,
                          reinterpret_cast<uint8_t*>(epi_stage) + quarter * 32 * 128,
                          mb * 128 + quarter * 32, nb);
      else if constexpr (EPI == EPI_RELU2 && BN % 64 == 0) {
        if (p.c_tma)
          epi_store_tma_relu2<BN, T16>(p, &tmC, taddr,
                                       reinterpret_cast<uint8_t*>(epi_stage) + quarter * 32 * 128,
                                       mb * 128 + quarter * 32, nb);
        else
          epi_store_rows<BN, T16>(p, taddr, epi_stage + quarter * 32 * C::kEpiStride,
                                  mb * 128 + quarter * 32, nb, EPI);
      }
      else
        epi_store_rows<BN, T16>(p, taddr, epi_stage + quarter * 32 * C::kEpiStride,
                                mb * 128 + quarter * 32, nb, EPI);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    // the staging area must outlive the reads of the last bulk stores
    if ((EPI == EPI_F32 || EPI == EPI_RELU2) && p.c_tma && lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}


// ======================================================================= host
// Status word of the single-step entry point (timeouts of a bare GEMM call).
__device__ uint32_t g_op_status;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <class T16> struct MapType;
template <> struct MapType<bf16> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; };
template <> struct MapType<f16> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; };
template <> struct MapType<e4m3> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_UINT8; };

// Row-major matrix [rows, cols] of 16- or 8-bit elements viewed as 2D (x =
// column, y = row); box of 128 bytes of columns (the swizzle width: 64 16-bit or
// 128 8-bit elements) by box_rows rows.
template <class T16>
static bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * sizeof(T16)};
  cuuint32_t box[2] = {128 / (uint32_t)sizeof(T16), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, MapType<T16>::v, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 matrix [rows, cols] with row pitch ld (elements) as the target of the
// epilogue's TMA stores: boxes of 32 x 32 values, 128-byte swizzle. Needs a 16-byte
// aligned base and ld % 4 == 0 (the caller falls back to plain stores otherwise).
static bool make_store_map(CUtensorMap* map, float* base, uint64_t rows, uint64_t cols, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) || (ld % 4) || cols == 0 || rows == 0)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 16-bit matrix [rows, cols] (pitch cols) as the target of the ReLU^2 epilogue's
// TMA stores: boxes of 64 x 32 values (128-byte rows), 128-byte swizzle.
template <class T16>
static bool make_store_map16(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) || (cols % 8) || cols == 0 || rows == 0)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * sizeof(T16)};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, MapType<T16>::v, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct LayerMaps {
  CUtensorMap wq, wk, wv, wo, wfc, wproj;
};

struct TcModel {
  nc_config cfg;
  bool f16 = true;   // 16-bit type of operands, activations and KV cache
  int sm_count = 148;
  std::vector<LayerMaps> layers;
  CUtensorMap lm;
  void *xn, *att, *h, *xnl;
  size_t max_rows;
  uint32_t* status;
};

static int sm_count_now() {
  int dev = 0, n = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

template <int BN, int EPI, class T16>
static nc_status launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
                             const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b2,
                             const GemmArgs& args, int sm_count, cudaStream_t s,
                             const CUtensorMap* c_map = nullptr) {
  using C = TileCfg<BN>;
  auto kern = gemm_tc_kernel<BN, EPI, T16>;
  if (!ensure_dyn_smem((const void*)kern, C::kSmemBytes)) return NC_ERR_CUDA;
  const int units = args.num_m_blk * args.num_n_blk * args.k_splits;
  const int grid = args.stream_k ? sm_count : std::min(units, sm_count);
  CUtensorMap cm;
  memset(&cm, 0, sizeof(cm));
  if (c_map) cm = *c_map;
  GemmArgs a = args;
  a.c_tma = ((EPI == EPI_F32 || (EPI == EPI_RELU2 && BN % 64 == 0)) && c_map) ? 1 : 0;
  kern<<<grid, 192, C::kSmemBytes, s>>>(a0, a1, a2, b0, b1, b2, cm, a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

static GemmArgs base_args(int M, int N, int K, int BN, uint32_t* status) {
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.num_m_blk = (M + 127) / 128;
  a.num_n_blk = (N + BN - 1) / BN;
  a.num_k_blk = K / 64;
  a.k_splits = 1;
  a.k_per_split = a.num_k_blk;
  a.a_split0 = a.a_split1 = INT_MAX;
  a.b_split0 = a.b_split1 = INT_MAX;
  a.status = status;
  return a;
}

// tile mode: N tile 128 or 256. A 128 x 128 x 16 MMA reads 8 KB of shared
// memory every 64 cycles (the full 128 B/clock of an SM), a 128 x 256 x 16 one
// 12 KB every 128 cycles, so 256 wins unless 128 wastes clearly less of the last
// wave. NC_GEMM_BN=128|256 in the environment forces one (measurement).
static int pick_bn(int M, int N, int sm_count) {
  static int forced = -1;
  if (forced < 0) {
    const char* e = getenv("NC_GEMM_BN");
    forced = e ? atoi(e) : 0;
  }
  if (forced == 128 || forced == 256) return forced;
  const int mb = (M + 127) / 128;
  auto cost = [&](int bn) {
    const int units = mb * ((N + bn - 1) / bn);
    return (int64_t)((units + sm_count - 1) / sm_count) * bn;
  };
  return cost(128) * 4 < cost(256) * 3 ? 128 : 256;
}

template <int EPI, class T16>
static nc_status tile_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const CUtensorMap& b2, GemmArgs args, int BN, int sm_count,
                           cudaStream_t s, const CUtensorMap* c_map = nullptr) {
  args.num_n_blk = (args.N + BN - 1) / BN;
  if (BN == 256) return launch_gemm<256, EPI, T16>(a, a, a, b0, b1, b2, args, sm_count, s, c_map);
  return launch_gemm<128, EPI, T16>(a, a, a, b0, b1, b2, args, sm_count, s, c_map);
}

// swap mode: features (weight rows, A) x tokens (B), split over K
static void plan_splits(GemmArgs& a, int sm_count) {
  int splits = std::max(1, sm_count / a.num_m_blk);
  splits = std::min(splits, std::min(kMaxSplits, a.num_k_blk));
  a.k_per_split = (a.num_k_blk + splits - 1) / splits;
  a.k_splits = (a.num_k_blk + a.k_per_split - 1) / a.k_per_split;
}

static int swap_bn(int64_t M) { return M <= 32 ? 32 : (M <= 64 ? 64 : 128); }

template <class T16>
static nc_status swap_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
                           const void* act, int64_t M, int K, GemmArgs args, int sm_count,
                           cudaStream_t s) {
  const int BN = swap_bn(M);
  CUtensorMap b;
  if (!make_map<T16>(&b, act, (uint64_t)M, (uint64_t)K, BN)) return NC_ERR_CUDA;
  args.num_n_blk = 1;
  if (BN == 32) return launch_gemm<32, EPI_SWAP, T16>(a0, a1, a2, b, b, b, args, sm_count, s);
  if (BN == 64) return launch_gemm<64, EPI_SWAP, T16>(a0, a1, a2, b, b, b, args, sm_count, s);
  return launch_gemm<128, EPI_SWAP, T16>(a0, a1, a2, b, b, b, args, sm_count, s);
}

// split-K partial sums of Y^T = W X^T, written as part[split][token][feature]
template <class T16>
static nc_status swap_partials(TcModel* t, const CUtensorMap& w0, const CUtensorMap& w1,
                               const CUtensorMap& w2, int split0, int split1, int n_feat, int K,
                               const void* act, int64_t M, float* part, int* n_split,
                               cudaStream_t s) {
  GemmArgs a = base_args(n_feat, (int)M, K, swap_bn(M), t->status);
  a.a_split0 = split0;
  a.a_split1 = split1;
  plan_splits(a, t->sm_count);
  a.out_f32 = part;
  a.ldo = n_feat;
  a.split_stride = (int64_t)M * n_feat;
  *n_split = a.k_splits;
  return swap_gemm<T16>(w0, w1, w2, act, M, K, a, t->sm_count, s);
}

static nc_dtype act_of(const TcModel* t) { return t->f16 ? NC_F16 : NC_BF16; }

template <class T16>
static nc_status qkv_impl(TcModel* t, int l, int64_t M, const RowMap& rm, const QkvDst& dst,
                          float* part, cudaStream_t s) {
  const nc_config& c = t->cfg;
  const LayerMaps& w = t->layers[l];
  const int d = c.d_model, qd = c.n_head * 128, kvd = c.n_kv_head * 128;
  const int nqkv = qd + 2 * kvd;
  if (M <= kSwapMaxRows) {
    int ns = 1;
    nc_status st = swap_partials<T16>(t, w.wq, w.wk, w.wv, qd, qd + kvd, nqkv, d, t->xn, M, part,
                                      &ns, s);
    if (st != NC_OK) return st;
    launch_qkv_post(part, ns, M, rm, dst, act_of(t), s);
    return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
  }
  CUtensorMap a;
  if (!make_map<T16>(&a, t->xn, (uint64_t)M, d, 128)) return NC_ERR_CUDA;
  GemmArgs args = base_args((int)M, nqkv, d, 256, t->status);
  args.b_split0 = qd;
  args.b_split1 = qd + kvd;
  args.rm = rm;
  args.qkv = dst;
  return launch_gemm<256, EPI_QKV, T16>(a, a, a, w.wq, w.wk, w.wv, args, t->sm_count, s);
}

template <class T16>
static nc_status out_proj_impl(TcModel* t, int l, int64_t M, float* x, float* part,
                               cudaStream_t s) {
  const nc_config& c = t->cfg;
  const LayerMaps& w = t->layers[l];
  const int d = c.d_model, qd = c.n_head * 128;
  if (M <= kSwapMaxRows) {
    int ns = 1;
    nc_status st = swap_partials<T16>(t, w.wo, w.wo, w.wo, INT_MAX, INT_MAX, d, qd, t->att, M,
                                      part, &ns, s);
    if (st != NC_OK) return st;
    launch_residual_finish(part, ns, x, M, d, nullptr, act_of(t), c.rms_eps, s);
    return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
  }
  CUtensorMap a;
  if (!make_map<T16>(&a, t->att, (uint64_t)M, qd, 128)) return NC_ERR_CUDA;
  const int BN = pick_bn((int)M, d, t->sm_count);
  GemmArgs args = base_args((int)M, d, qd, BN, t->status);
  args.out_f32 = x;
  args.ldo = d;
  args.stream_k = 1;
  return tile_gemm<EPI_RESID, T16>(a, w.wo, w.wo, w.wo, args, BN, t->sm_count, s);
}

template <class T16>
static nc_status fc_impl(TcModel* t, int l, int64_t M, float* part, cudaStream_t s) {
  const nc_config& c = t->cfg;
  const LayerMaps& w = t->layers[l];
  const int d = c.d_model, F = c.d_mlp;
  if (M <= kSwapMaxRows) {
    int ns = 1;
    nc_status st = swap_partials<T16>(t, w.wfc, w.wfc, w.wfc, INT_MAX, INT_MAX, F, d, t->xn, M,
                                      part, &ns, s);
    if (st != NC_OK) return st;
    launch_relu2_finish(part, ns, t->h, M, F, act_of(t), t->status, s);
    return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
  }
  CUtensorMap a;
  if (!make_map<T16>(&a, t->xn, (uint64_t)M, d, 128)) return NC_ERR_CUDA;
  const int BN = pick_bn((int)M, F, t->sm_count);
  GemmArgs args = base_args((int)M, F, d, BN, t->status);
  args.out_16 = t->h;
  args.ldo = F;
  CUtensorMap hmap;
  const bool tma = make_store_map16<T16>(&hmap, t->h, (uint64_t)M, F);
  return tile_gemm<EPI_RELU2, T16>(a, w.wfc, w.wfc, w.wfc, args, BN, t->sm_count, s,
                                   tma ? &hmap : nullptr);
}

template <class T16>
static nc_status proj_impl(TcModel* t, int l, int64_t M, float* x, float* part, cudaStream_t s) {
  const nc_config& c = t->cfg;
  const LayerMaps& w = t->layers[l];
  const int d = c.d_model, F = c.d_mlp;
  if (M <= kSwapMaxRows) {
    int ns = 1;
    nc_status st = swap_partials<T16>(t, w.wproj, w.wproj, w.wproj, INT_MAX, INT_MAX, d, F, t->h,
                                      M, part, &ns, s);
    if (st != NC_OK) return st;
    launch_residual_finish(part, ns, x, M, d, nullptr, act_of(t), c.rms_eps, s);
    return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
  }
  CUtensorMap a;
  if (!make_map<T16>(&a, t->h, (uint64_t)M, F, 128)) return NC_ERR_CUDA;
  const int BN = pick_bn((int)M, d, t->sm_count);
  GemmArgs args = base_args((int)M, d, F, BN, t->status);
  args.out_f32 = x;
  args.ldo = d;
  args.stream_k = 1;
  // A (M x F, 16-bit) larger than about half of L2: group the CTAs by n block
  // when at most 3% of the SMs would stay idle
  const int G = args.num_n_blk;
  if ((int64_t)M * F * 2 > (int64_t)48 << 20 && G > 1 && G <= t->sm_count &&
      (t->sm_count % G) * 100 <= 3 * t->sm_count)
    args.sk_groups = G;
  return tile_gemm<EPI_RESID, T16>(a, w.wproj, w.wproj, w.wproj, args, BN, t->sm_count, s);
}

template <class T16>
static nc_status lm_impl(TcModel* t, const void* xn, int64_t M, float* logits, cudaStream_t s) {
  const nc_config& c = t->cfg;
  const int d = c.d_model, V = c.vocab;
  if (M <= kSwapMaxRows) {
    GemmArgs a = base_args(V, (int)M, d, swap_bn(M), t->status);
    a.out_f32 = logits;
    a.ldo = V;
    a.split_stride = 0;
    return swap_gemm<T16>(t->lm, t->lm, t->lm, xn, M, d, a, t->sm_count, s);
  }
  CUtensorMap a;
  if (!make_map<T16>(&a, xn, (uint64_t)M, d, 128)) return NC_ERR_CUDA;
  GemmArgs args = base_args((int)M, V, d, 256, t->status);
  args.out_f32 = logits;
  args.ldo = V;
  CUtensorMap cmap;
  const bool tma = make_store_map(&cmap, logits, (uint64_t)M, V, V);
  return tile_gemm<EPI_F32, T16>(a, t->lm, t->lm, t->lm, args, 256, t->sm_count, s,
                                 tma ? &cmap : nullptr);
}

template <class T16>
static bool build_maps(TcModel* t, const void* lm_head, const void* const* wq,
                       const void* const* wk, const void* const* wv, const void* const* wo,
                       const void* const* w_fc, const void* const* w_proj) {
  const nc_config& cfg = t->cfg;
  const uint64_t d = cfg.d_model, qd = (uint64_t)cfg.n_head * 128,
                 kvd = (uint64_t)cfg.n_kv_head * 128, F = cfg.d_mlp;
  t->layers.resize(cfg.n_layer);
  bool ok = make_map<T16>(&t->lm, lm_head, cfg.vocab, d, 128);
  for (int l = 0; l < cfg.n_layer && ok; ++l) {
    LayerMaps& m = t->layers[l];
    ok = make_map<T16>(&m.wq, wq[l], qd, d, 128) && make_map<T16>(&m.wk, wk[l], kvd, d, 128) &&
         make_map<T16>(&m.wv, wv[l], kvd, d, 128) && make_map<T16>(&m.wo, wo[l], d, qd, 128) &&
         make_map<T16>(&m.wfc, w_fc[l], F, d, 128) && make_map<T16>(&m.wproj, w_proj[l], d, F, 128);
  }
  return ok;
}

nc_status tc_create(const nc_config& cfg, const void* lm_head, const void* const* wq,
                    const void* const* wk, const void* const* wv, const void* const* wo,
                    const void* const* w_fc, const void* const* w_proj, void* xn, void* att,
                    void* h, void* xnl, size_t max_rows, uint32_t* status, TcModel** out) {
  if (!encode_fn()) return NC_ERR_CUDA;
  TcModel* t = new TcModel();
  t->cfg = cfg;
  t->f16 = cfg.act_dtype == NC_F16;
  t->sm_count = sm_count_now();
  t->xn = xn;
  t->att = att;
  t->h = h;
  t->xnl = xnl;
  t->max_rows = max_rows;
  t->status = status;
  const bool ok = t->f16 ? build_maps<f16>(t, lm_head, wq, wk, wv, wo, w_fc, w_proj)
                         : build_maps<bf16>(t, lm_head, wq, wk, wv, wo, w_fc, w_proj);
  if (!ok) {
    delete t;
    return NC_ERR_CUDA;
  }
  *out = t;
  return NC_OK;
}

void tc_destroy(TcModel* t) { delete t; }

nc_status tc_qkv(TcModel* t, int l, int64_t M, const RowMap& rm, const QkvDst& dst, float* part,
                 cudaStream_t s) {
  return t->f16 ? qkv_impl<f16>(t, l, M, rm, dst, part, s) : qkv_impl<bf16>(t, l, M, rm, dst, part, s);
}
nc_status tc_out_proj(TcModel* t, int l, int64_t M, float* x, float* part, cudaStream_t s) {
  return t->f16 ? out_proj_impl<f16>(t, l, M, x, part, s) : out_proj_impl<bf16>(t, l, M, x, part, s);
}
nc_status tc_fc(TcModel* t, int l, int64_t M, float* part, cudaStream_t s) {
  return t->f16 ? fc_impl<f16>(t, l, M, part, s) : fc_impl<bf16>(t, l, M, part, s);
}
nc_status tc_proj(TcModel* t, int l, int64_t M, float* x, float* part, cudaStream_t s) {
  return t->f16 ? proj_impl<f16>(t, l, M, x, part, s) : proj_impl<bf16>(t, l, M, x, part, s);
}
nc_status tc_lm_head(TcModel* t, const void* xn, int64_t M, float* logits, float* part,
                     cudaStream_t s) {
  (void)part;
  return t->f16 ? lm_impl<f16>(t, xn, M, logits, s) : lm_impl<bf16>(t, xn, M, logits, s);
}

// The LM head's 128 x 256 tiles reduced in the epilogue to the softmax partials
// of each (row, n block) and the target logits; tile mode for every M.
template <class T16>
static nc_status lm_loss_impl(TcModel* t, const void* xn, int64_t M, const int32_t* targets,
                              float2* part, float* zt, cudaStream_t s) {
  const nc_config& c = t->cfg;
  CUtensorMap a;
  if (!make_map<T16>(&a, xn, (uint64_t)M, c.d_model, 128)) return NC_ERR_CUDA;
  GemmArgs args = base_args((int)M, c.vocab, c.d_model, 256, t->status);
  args.out_f32 = reinterpret_cast<float*>(part);
  args.targets = targets;
  args.ce_zt = zt;
  return tile_gemm<EPI_CE, T16>(a, t->lm, t->lm, t->lm, args, 256, t->sm_count, s);
}

int lm_loss_blocks(int vocab) { return (vocab + 255) / 256; }

nc_status tc_lm_loss(TcModel* t, const void* xn, int64_t M, const int32_t* targets, float2* part,
                     float* zt, cudaStream_t s) {
  return t->f16 ? lm_loss_impl<f16>(t, xn, M, targets, part, zt, s)
                : lm_loss_impl<bf16>(t, xn, M, targets, part, zt, s);
}

// ------------------------------------------------- fp8 (E4M3) projections
static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// One CTA per row: scale = max|x[r, :]| / 448 (1 for a zero row) and the codes
// E4M3(x / scale), rounded to nearest even and saturating, two per conversion.
// The division is IEEE (the rounding decision matches a float32 reference).
template <class TI>
__global__ void quantize_e4m3_kernel(const TI* __restrict__ x, int64_t rows, int cols,
                                     uint8_t* __restrict__ q, float* __restrict__ scale) {
  __shared__ float red[32];
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  const TI* xr = x + r * cols;
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(to_f32(xr[c])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  amax = red[0];
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) scale[r] = s;
  uint8_t* qr = q + r * cols;
  for (int c = 2 * threadIdx.x; c < cols; c += 2 * blockDim.x) {
    const float a = __fdiv_rn(to_f32(xr[c]), s), b = __fdiv_rn(to_f32(xr[c + 1]), s);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(qr + c) =
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  }
}

nc_status quantize_e4m3(const void* x, nc_dtype dt, int64_t rows, int cols, uint8_t* q, float* scale,
                        cudaStream_t s) {
  if (rows == 0) return NC_OK;
  const dim3 grid((unsigned)rows), block(256);
  if (dt == NC_F32)
    quantize_e4m3_kernel<float><<<grid, block, 0, s>>>((const float*)x, rows, cols, q, scale);
  else if (dt == NC_BF16)
    quantize_e4m3_kernel<bf16><<<grid, block, 0, s>>>((const bf16*)x, rows, cols, q, scale);
  else
    quantize_e4m3_kernel<f16><<<grid, block, 0, s>>>((const f16*)x, rows, cols, q, scale);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

size_t gemv_e4m3_scratch_bytes(int N, int K, int B) {
  const int BN = swap_bn(B);
  const size_t xq = align256((size_t)BN * K), xs = 512;
  const size_t part = (size_t)kMaxSplits * B * N * 4;
  return xq + xs + part;
}

// y[t, n] = w_scale[n] * s_t * sum_k wq[n, k] * E4M3(x[t, k] / s_t): the activations
// are quantised per token into the scratch, then the swap-mode tcgen05 GEMM
// (kind::f8f6f4, features as M, tokens as N, split over K) writes scaled partial
// sums that one pass adds.
nc_status gemv_e4m3(const uint8_t* wq, const float* w_scale, int N, int K, const float* x, int B,
                    float* y, void* scratch, cudaStream_t s) {
  const int BN = swap_bn(B);
  uint8_t* xq = static_cast<uint8_t*>(scratch);
  float* xs = reinterpret_cast<float*>(xq + align256((size_t)BN * K));
  float* part = xs + 128;
  // token rows past B are read by the tile: zero codes
  if (BN > B && cudaMemsetAsync(xq + (size_t)B * K, 0, (size_t)(BN - B) * K, s) != cudaSuccess)
    return NC_ERR_CUDA;
  nc_status st = quantize_e4m3(x, NC_F32, B, K, xq, xs, s);
  if (st != NC_OK) return st;
  CUtensorMap a, b;
  if (!make_map<e4m3>(&a, wq, (uint64_t)N, (uint64_t)K, 128) ||
      !make_map<e4m3>(&b, xq, (uint64_t)BN, (uint64_t)K, BN))
    return NC_ERR_CUDA;
  const int sm = sm_count_now();
  GemmArgs args = base_args(N, B, K, BN, nullptr);
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&args.status), g_op_status) != cudaSuccess)
    return NC_ERR_CUDA;
  args.num_k_blk = K / 128;   // 128 one-byte elements per 128-byte row of a stage
  args.k_per_split = args.num_k_blk;
  plan_splits(args, sm);
  args.num_n_blk = 1;
  args.out_f32 = part;
  args.ldo = N;
  args.split_stride = (int64_t)B * N;
  args.row_scale = w_scale;
  args.tok_scale = xs;
  if (BN == 32)
    st = launch_gemm<32, EPI_SWAP, e4m3>(a, a, a, b, b, b, args, sm, s);
  else if (BN == 64)
    st = launch_gemm<64, EPI_SWAP, e4m3>(a, a, a, b, b, b, args, sm, s);
  else
    st = launch_gemm<128, EPI_SWAP, e4m3>(a, a, a, b, b, b, args, sm, s);
  if (st != NC_OK) return st;
  launch_sum_splits(part, args.k_splits, y, B, N, N, s);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status tc_cross_entropy(const void* A, const void* B, const int32_t* targets, int M, int N,
                           int K, nc_dtype dt, float2* part, float* zt, cudaStream_t s) {
  CUtensorMap a, b;
  const bool h = dt == NC_F16;
  const bool ok = h ? (make_map<f16>(&a, A, M, K, 128) && make_map<f16>(&b, B, N, K, 128))
                    : (make_map<bf16>(&a, A, M, K, 128) && make_map<bf16>(&b, B, N, K, 128));
  if (!ok) return NC_ERR_CUDA;
  const int sm = sm_count_now();
  GemmArgs args = base_args(M, N, K, 256, nullptr);
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&args.status), g_op_status) != cudaSuccess)
    return NC_ERR_CUDA;
  args.out_f32 = reinterpret_cast<float*>(part);
  args.targets = targets;
  args.ce_zt = zt;
  return h ? tile_gemm<EPI_CE, f16>(a, b, b, b, args, 256, sm, s)
           : tile_gemm<EPI_CE, bf16>(a, b, b, b, args, 256, sm, s);
}

nc_status tc_gemm_f32out(const void* A, const void* B, float* C, int M, int N, int K,
                         nc_dtype dt, cudaStream_t s) {
  CUtensorMap a, b;
  const bool h = dt == NC_F16;
  const bool ok = h ? (make_map<f16>(&a, A, M, K, 128) && make_map<f16>(&b, B, N, K, 128))
                    : (make_map<bf16>(&a, A, M, K, 128) && make_map<bf16>(&b, B, N, K, 128));
  if (!ok) return NC_ERR_CUDA;
  const int sm = sm_count_now();
  const int BN = pick_bn(M, N, sm);
  GemmArgs args = base_args(M, N, K, BN, nullptr);
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&args.status), g_op_status) != cudaSuccess)
    return NC_ERR_CUDA;
  args.out_f32 = C;
  args.ldo = N;
  CUtensorMap cmap;
  const CUtensorMap* cm = make_store_map(&cmap, C, M, N, N) ? &cmap : nullptr;
  return h ? tile_gemm<EPI_F32, f16>(a, b, b, b, args, BN, sm, s, cm)
           : tile_gemm<EPI_F32, bf16>(a, b, b, b, args, BN, sm, s, cm);
}

}  // namespace nc
