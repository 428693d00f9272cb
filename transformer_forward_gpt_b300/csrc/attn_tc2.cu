// Causal flash attention for prefill on tcgen05, two query tiles per CTA
// (head_dim 128, 16-bit Q/K/V, fp32 softmax and accumulation in TMEM).
//
// CTA = 256 queries (query tiles A and B, 128 each) of one (sequence, query
// head); 320 threads:
//   warp 0      TMA: Q_A and Q_B once, then K and V tiles of 128 keys into
//               two-slot rings (keys at or past T read as zeros)
//   warp 1      TMEM owner; one thread issues, per key tile j,
//               S_A = Q_A K^T, S_B = Q_B K^T into two TMEM score buffers and
//               O_X += P_X V with P_X read from TMEM (the A operand of a
//               tcgen05.mma may live in tensor memory)
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B: thread = query
//               = TMEM lane. A thread reads its score row in 32-column chunks
//               (row max first, then 2^(s - m)), and writes the 16-bit P row
//               back over the first 64 columns of its own score buffer.
// The MMA issue order S_A(j+1) after P_A(j) V, S_B(j+1) after P_B(j) V lets
// tile B's softmax run while tile A's matrix products do and vice versa; since
// tcgen05.mma operations of one thread complete in issue order, "S_X(j) done"
// also means "P_X(j-1) V done", so P may overwrite the score buffer and O may
// be rescaled without another barrier. The exponent's reference max is raised
// only when a row's max grows by more than 8 (log2 units), as in the one-tile
// kernel.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc.h"

namespace nc {
namespace {

constexpr int kHd = 128;
constexpr int kBq = 128;
constexpr int kBk = 128;
constexpr int kTile = 128 * 128 * 2;
constexpr int kHalf = kTile / 2;
constexpr int kOffQA = 0, kOffQB = kTile, kOffK = 2 * kTile, kOffV = 4 * kTile, kOffBar = 6 * kTile;
constexpr size_t kSmem = 6 * kTile + 256 + 1024;
__device__ __forceinline__ uint32_t col_s(int x) { return (uint32_t)x * 128u; }          // scores / P
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + (uint32_t)x * 128u; }   // output
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// D(tmem) (+)= A(tmem) * B(smem desc)^T, 16-bit inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16kind_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

struct Attn2Args {
  int B, H, Hkv, T, n_qt, n_qp;
  float scale_log2;
  void* o;
  uint32_t* status;
};

template <class T16>
__global__ void __launch_bounds__(320, 1)
    attn_prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const Attn2Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;          // 1
  uint64_t* k_full = bars + 1;      // 2
  uint64_t* k_empty = bars + 3;     // 2
  uint64_t* v_full = bars + 5;      // 2
  uint64_t* v_empty = bars + 7;     // 2
  uint64_t* s_full = bars + 9;      // [tile A, tile B]
  uint64_t* p_full = bars + 11;     // [tile A, tile B], 4 warps each
  uint64_t* o_done = bars + 13;     // every MMA of the CTA done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);

  const int per_qp = a.B * a.H;
  const int qp = a.n_qp - 1 - (int)(blockIdx.x / per_qp);   // heaviest pairs first
  const int bh = (int)(blockIdx.x % per_qp);
  const int b = bh / a.H, h = bh % a.H;
  const int g = h / (a.H / a.Hkv);
  const int qt[2] = {2 * qp, 2 * qp + 1};
  const int nk[2] = {qt[0] + 1, qt[1] < a.n_qt ? qt[1] + 1 : 0};   // key tiles per query tile
  const int n_kt = nk[1] > nk[0] ? nk[1] : nk[0];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(o_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int nq = nk[1] > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq * kTile);
      for (int x = 0; x < nq; ++x) {
        uint8_t* qd = smem + (x == 0 ? kOffQA : kOffQB);
        tma_load_3d(qd, &tmQ, q_full, 0, qt[x] * kBq, bh);
        tma_load_3d(qd + kHalf, &tmQ, q_full, 64, qt[x] * kBq, bh);
      }
      const int bg = b * a.Hkv + g;
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        const uint32_t par = ((j >> 1) & 1) ^ 1;
        if (!mbar_wait(&k_empty[st], par, a.status)) break;
        uint8_t* kd = smem + kOffK + st * kTile;
        mbar_arrive_expect_tx(&k_full[st], kTile);
        tma_load_4d(kd, &tmK, &k_full[st], 0, j * kBk, bg, 0);
        tma_load_4d(kd + kHalf, &tmK, &k_full[st], 64, j * kBk, bg, 0);
        ++issued_k;
        if (!mbar_wait(&v_empty[st], par, a.status)) break;
        uint8_t* vd = smem + kOffV + st * kTile;
        mbar_arrive_expect_tx(&v_full[st], kTile);
        tma_load_4d(vd, &tmV, &v_full[st], 0, j * kBk, bg, 0);
        tma_load_4d(vd + kHalf, &tmV, &v_full[st], 64, j * kBk, bg, 0);
        ++issued_v;
      }
      // copies in flight must land before shared memory is released
      mbar_wait(q_full, 0, a.status);
      for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j)
        mbar_wait(&k_full[j & 1], (j >> 1) & 1, a.status);
      for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j)
        mbar_wait(&v_full[j & 1], (j >> 1) & 1, a.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdS = idesc_f32acc(Fmt16<T16>::code, 128, 128);
      constexpr uint32_t kIdO = idesc_f32acc(Fmt16<T16>::code, 128, 128) | (1u << 16);  // B MN-major
      const uint32_t sQ[2] = {smem_u32(smem + kOffQA), smem_u32(smem + kOffQB)};
      bool ok = mbar_wait(q_full, 0, a.status);
      auto issue_s = [&](int x, int j) {
        const uint32_t sK = smem_u32(smem + kOffK + (j & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t da = sdesc_kmajor_sw128(sQ[x] + (kk >> 2) * kHalf + (kk & 3) * 32);
          const uint64_t db = sdesc_kmajor_sw128(sK + (kk >> 2) * kHalf + (kk & 3) * 32);
          mma_f16kind_ss(tmem + col_s(x), da, db, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[x]);
      };
      auto issue_pv = [&](int x, int j) {
        const uint32_t sV = smem_u32(smem + kOffV + (j & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // P columns: keys 16kk..16kk+15 are 8 packed 32-bit columns
          const uint64_t db = sdesc_mn_sw128(sV + kk * 16 * 128, kHalf);
          mma_f16kind_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8, db, kIdO,
                         (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      // prologue: scores of key tile 0 for both query tiles
      if (ok) ok = mbar_wait(&k_full[0], 0, a.status);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (nk[1] > 0) issue_s(1, 0);
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; j < n_kt && ok; ++j) {
        const int jn = j + 1;
        if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1, a.status)) {
          ok = false;
          break;
        }
        const bool need_k = jn < nk[0] || jn < nk[1];
        bool k_ready = false;
        for (int x = 0; x < 2 && ok; ++x) {
          if (j < nk[x]) {
            if (!mbar_wait(&p_full[x], j & 1, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(x, j);
          }
          if (jn < nk[x]) {
            if (!k_ready) {
              if (!mbar_wait(&k_full[jn & 1], (jn >> 1) & 1, a.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_ready = true;
            }
            issue_s(x, jn);
          }
        }
        if (!ok) break;
        if (need_k) mma_commit(&k_empty[jn & 1]);
        mma_commit(&v_empty[j & 1]);
      }
      if (ok) mma_commit(o_done);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int x = (warp - 2) / 4;            // query tile of this group
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;    // = TMEM lane
    const int qpos = qt[x] * kBq + row;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_col = tmem + lane_base + col_s(x);
    const uint32_t o_col = tmem + lane_base + col_o(x);
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < nk[x]; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      const bool diag = j == qt[x];
      const int kmax = qpos - j * kBk;
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32_sync(s_col + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          mx = fmaxf(mx, (diag && c * 32 + i > kmax) ? -INFINITY : v[i] * a.scale_log2);
      }
      const bool raise = mx > m_ref + 8.f;
      const float m_new = raise ? mx : m_ref;
      const float corr = raise ? exp2f(m_ref - m_new) : 1.f;
      float psum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32_sync(s_col + c * 32, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int i0 = c * 32 + 2 * i;
          const float p0 = (diag && i0 > kmax) ? 0.f : ex2_approx(fmaf(v[2 * i], a.scale_log2, -m_new));
          const float p1 = (diag && i0 + 1 > kmax) ? 0.f : ex2_approx(fmaf(v[2 * i + 1], a.scale_log2, -m_new));
          psum += p0 + p1;
          pk[c * 16 + i] = pack2<T16>(p0, p1);
        }
      }
      l_sum = l_sum * corr + psum;
      m_ref = m_new;
      // S_X(j) done implies P_X(j-1) V done: O_X may be rescaled, P may be written
      if (j >= 1 && __any_sync(0xffffffffu, raise)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32_sync(o_col + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= corr;
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
          tmem_st32(o_col + c * 32, w);
        }
      }
      {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[i];
        tmem_st32(s_col, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[32 + i];
        tmem_st32(s_col + 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok && nk[x] > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done, 0, a.status));
    if (ok && nk[x] > 0) {
      tc_fence_after();
      // O / l -> out[b, qpos, h*128 ..], staged through this warp's rows of the
      // tile's (idle) Q buffer, 256-byte rows with 16-byte chunks XOR-swizzled
      const float inv = 1.f / l_sum;
      uint8_t* stage = smem + (x == 0 ? kOffQA : kOffQB) + quarter * 32 * 256;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32_sync(o_col + c * 32, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int chunk = c * 4 + i;
          *reinterpret_cast<uint4*>(stage + lane * 256 + ((chunk ^ (lane & 15)) << 4)) =
              make_uint4(pack2<T16>(v[8 * i] * inv, v[8 * i + 1] * inv),
                         pack2<T16>(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                         pack2<T16>(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                         pack2<T16>(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        }
      }
      __syncwarp();
      T16* out = static_cast<T16*>(a.o);
#pragma unroll 1
      for (int it = 0; it < 16; ++it) {
        const int r = it * 2 + lane / 16, cc = lane % 16;
        const int t = qt[x] * kBq + quarter * 32 + r;
        if (t < a.T)
          *reinterpret_cast<uint4*>(out + ((int64_t)b * a.T + t) * (a.H * kHd) + h * kHd + cc * 8) =
              *reinterpret_cast<const uint4*>(stage + r * 256 + ((cc ^ (r & 15)) << 4));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Same contract as tc_attention_prefill_tc, with prebuilt tensor maps.
nc_status attn2_launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       void* o, int B, int H, int Hkv, int T, bool half, uint32_t* status,
                       cudaStream_t s) {
  Attn2Args a;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.T = T;
  a.n_qt = (T + kBq - 1) / kBq;
  a.n_qp = (a.n_qt + 1) / 2;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kHd));
  a.o = o;
  a.status = status;
  const unsigned grid = (unsigned)(a.n_qp * B * H);
  if (half) {
    static bool cfg = false;
    if (!cfg) {
      if (cudaFuncSetAttribute(attn_prefill_tc2_kernel<f16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return NC_ERR_CUDA;
      cfg = true;
    }
    attn_prefill_tc2_kernel<f16><<<grid, 320, kSmem, s>>>(mq, mk, mv, a);
  } else {
    static bool cfg = false;
    if (!cfg) {
      if (cudaFuncSetAttribute(attn_prefill_tc2_kernel<bf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return NC_ERR_CUDA;
      cfg = true;
    }
    attn_prefill_tc2_kernel<bf16><<<grid, 320, kSmem, s>>>(mq, mk, mv, a);
  }
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace nc
