// Causal flash attention for prefill on tcgen05 (head_dim 128, 16-bit Q/K/V,
// fp32 softmax and accumulation in TMEM), with grouped-query head sharing.
//
// CTA = 128 queries of one (sequence, query head); 320 threads:
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into a
//               two-stage ring (keys at or past T read as zeros)
//   warp 1      TMEM owner; one thread issues S = Q K^T (M = N = K = 128) into
//               one of two TMEM score buffers, and O += P V (P from shared
//               memory, V as an MN-major operand) into the TMEM output
//   warps 2..9  softmax: warps w and w + 4 share the TMEM lane quarter w % 4
//               (thread = query row) and split the row's 128 key columns in two
//               halves; the pair exchanges row maxima through shared memory.
//               A thread masks keys past the query on the diagonal tile,
//               exponentiates in the log2 domain and writes its half of the P
//               row (16-bit) to shared memory.
// The running max used as the exponent's reference is only raised when a row's
// max grows by more than 8 (log2 units): then that row of O is rescaled in TMEM.
// Otherwise p <= 2^8 and the reference stays, which keeps O in TMEM untouched
// on almost every tile; the final O / l is the same either way. Scores of tile
// j+1 are computed while the softmax of tile j runs.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc.h"

namespace nc {

nc_status attn2_launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       void* o, int B, int H, int Hkv, int T, bool half, uint32_t* status,
                       cudaStream_t s);

namespace {

constexpr int kHd = 128;
constexpr int kBq = 128;            // queries per CTA
constexpr int kBk = 128;            // keys per tile
constexpr int kTile = 128 * 128 * 2;   // 32 KB: a 128 x 128 16-bit tile (two 64-column boxes)
constexpr int kHalf = kTile / 2;

// shared memory: Q | K[2] | V[2] | P | barriers
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;
constexpr int kOffV = 3 * kTile;
constexpr int kOffP = 5 * kTile;
constexpr int kOffBar = 6 * kTile;
constexpr int kOffX = 6 * kTile + 256;        // [2 parity][128 rows][2 halves] row maxima
constexpr int kOffL = kOffX + 2048;           // [128 rows][2 halves] final row sums
constexpr size_t kSmem = 6 * kTile + 256 + 3072 + 1024;

// TMEM columns: S[0] 0..127, S[1] 128..255, O 256..383
constexpr uint32_t kColS0 = 0, kColO = 256, kTmemCols = 512;

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

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 64 MN values per 128-byte row, K rows 128 bytes apart in 1 KB atoms (SBO),
// the next 64 MN values `lbo` bytes further (LBO).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st32_sync(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

// byte offset of 16-byte chunk c (0..15) of row r in a 128-row tile stored as
// two 64-column boxes with the 128-byte swizzle
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct AttnArgs {
  int B, H, Hkv, T, n_qt;
  float scale_log2;
  void* o;            // [B, T, H*128]
  uint32_t* status;
};

template <class T16>
__global__ void __launch_bounds__(320, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const AttnArgs a, int layer) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;          // 1
  uint64_t* k_full = bars + 1;      // 2
  uint64_t* k_empty = bars + 3;     // 2 (freed once S of the tile is done)
  uint64_t* v_full = bars + 5;      // 2
  uint64_t* v_empty = bars + 7;     // 2 (freed once P V of the tile is done)
  uint64_t* s_full = bars + 9;      // 2
  uint64_t* s_free = bars + 11;     // 2 (4 softmax warps)
  uint64_t* p_full = bars + 13;     // 1 (4 softmax warps)
  uint64_t* o_done = bars + 14;     // 1 (one commit per P V)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);
  // [quarter][3]: the two softmax warps of a lane quarter exchange row maxima
  // (slots 0, 1 by tile parity) and the final row sums (slot 2); 2 arrivals each
  uint64_t* xbar = bars + 18;

  // heaviest query tiles first
  const int per_qt = a.B * a.H;
  const int qt = a.n_qt - 1 - (int)(blockIdx.x / per_qt);
  const int bh = (int)(blockIdx.x % per_qt);
  const int b = bh / a.H, h = bh % a.H;
  const int g = h / (a.H / a.Hkv);
  const int n_kt = qt + 1;   // key tiles 0..qt (causal)

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 8);
    }
    mbar_init(p_full, 8);
    mbar_init(o_done, 1);
    for (int i = 0; i < 12; ++i) mbar_init(&xbar[i], 2);
    *abort_flag = 0;
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
      mbar_arrive_expect_tx(q_full, kTile);
      tma_load_3d(smem + kOffQ, &tmQ, q_full, 0, qt * kBq, bh);
      tma_load_3d(smem + kOffQ + kHalf, &tmQ, q_full, 64, qt * kBq, bh);
      const int bg = b * a.Hkv + g;
      int issued = 0;
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        const uint32_t par = ((j >> 1) & 1) ^ 1;
        if (!mbar_wait(&k_empty[st], par, a.status)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* kd = smem + kOffK + st * kTile;
        mbar_arrive_expect_tx(&k_full[st], kTile);
        tma_load_4d(kd, &tmK, &k_full[st], 0, j * kBk, bg, layer);
        tma_load_4d(kd + kHalf, &tmK, &k_full[st], 64, j * kBk, bg, layer);
        ++issued_k;
        if (!mbar_wait(&v_empty[st], par, a.status)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* vd = smem + kOffV + st * kTile;
        mbar_arrive_expect_tx(&v_full[st], kTile);
        tma_load_4d(vd, &tmV, &v_full[st], 0, j * kBk, bg, layer);
        tma_load_4d(vd + kHalf, &tmV, &v_full[st], 64, j * kBk, bg, layer);
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
      const uint32_t sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP);
      bool ok = mbar_wait(q_full, 0, a.status);
      auto pv = [&](int jj) -> bool {
        // O (+)= P V_jj once the softmax has written P_jj
        if (!mbar_wait(p_full, jj & 1, a.status) ||
            !mbar_wait(&v_full[jj & 1], (jj >> 1) & 1, a.status))
          return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + kOffV + (jj & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // keys 16kk..16kk+15: P columns (K-major), V rows (MN-major)
          const uint64_t da = sdesc_kmajor_sw128(sP + (kk >> 2) * kHalf + (kk & 3) * 32);
          const uint64_t db = sdesc_mnmajor_sw128(sV + kk * 16 * 128, kHalf);
          mma_f16kind_ss(tmem + kColO, da, db, kIdO, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&v_empty[jj & 1]);
        return true;
      };
      for (int j = 0; j < n_kt && ok; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&k_full[st], (j >> 1) & 1, a.status) ||
            !mbar_wait(&s_free[st], ((j >> 1) & 1) ^ 1, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + kOffK + st * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t da = sdesc_kmajor_sw128(sQ + (kk >> 2) * kHalf + (kk & 3) * 32);
          const uint64_t db = sdesc_kmajor_sw128(sK + (kk >> 2) * kHalf + (kk & 3) * 32);
          mma_f16kind_ss(tmem + kColS0 + st * 128, da, db, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[st]);
        mma_commit(&k_empty[st]);
        if (j >= 1 && !pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) ok = pv(n_kt - 1);
      if (!ok) *abort_flag = 1;
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int quarter = warp % 4;
    const int half = (warp - 2) / 4;          // key / output columns [64 half, 64 half + 64)
    const int row = quarter * 32 + lane;      // query row within the tile = TMEM lane
    const int qpos = qt * kBq + row;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint8_t* sP = smem + kOffP;
    float* xch = reinterpret_cast<float*>(smem + kOffX);
    float* xl = reinterpret_cast<float*>(smem + kOffL);
    uint64_t* qbar = xbar + 3 * quarter;      // this quarter's exchange barriers
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int st = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[st], (j >> 1) & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      // this half of the score row in one 64-column TMEM load; causal mask
      const uint32_t s_col = tmem + lane_base + kColS0 + st * 128 + 64 * half;
      const bool diag = j == qt;
      const int kmax = qpos - j * kBk - 64 * half;   // keys i > kmax are masked (diagonal)
      float sv[64];
      tmem_ld64_sync(s_col, sv);
      if (diag) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i > kmax) sv[i] = -INFINITY;
      }
      // row max over both halves (raw scores; the scale > 0 is applied to the max
      // and folded into the exponent's FMA), exchanged through shared memory
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) mx = fmaxf(mx, sv[i]);
      xch[(st * 128 + row) * 2 + half] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&qbar[st]);
      ok = __all_sync(0xffffffffu, mbar_wait(&qbar[st], (j >> 1) & 1, a.status));
      if (!ok) break;
      mx = fmaxf(mx, xch[(st * 128 + row) * 2 + (half ^ 1)]) * a.scale_log2;
      // raise the reference only when the max outgrows it by 2^8
      const bool raise = mx > m_ref + 8.f;
      const float m_new = raise ? mx : m_ref;
      const float corr = raise ? ex2_approx(m_ref - m_new) : 1.f;   // 0 on the first tile
      // p = 2^(s - m) packed to 16 bits in registers, this half's row sum
      float psum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(fmaf(sv[2 * i], a.scale_log2, -m_new));
        const float p1 = ex2_approx(fmaf(sv[2 * i + 1], a.scale_log2, -m_new));
        psum += p0 + p1;
        pk[i] = pack2<T16>(p0, p1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[st]);
      l_sum = l_sum * corr + psum;
      m_ref = m_new;
      // P V of the previous tile must be done before P is overwritten or O touched
      if (j >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, a.status));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {   // this half of the O row
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float v[32];
            const uint32_t oc = tmem + lane_base + kColO + 64 * half + c * 32;
            tmem_ld32_sync(oc, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= corr;
            tmem_st32_sync(oc, v);
          }
        }
      }
      // this half of the P row -> shared memory (K-major, 128-byte swizzle)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sP + tile_off(row, 8 * half + c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_kt - 1) & 1, a.status));
    // the row sum is the two halves' sums (same reference max)
    if (ok) {
      xl[row * 2 + half] = l_sum;
      __syncwarp();
      if (lane == 0) mbar_arrive(&qbar[2]);
      ok = __all_sync(0xffffffffu, mbar_wait(&qbar[2], 0, a.status));
      if (ok) l_sum += xl[row * 2 + (half ^ 1)];
    }
    if (ok) {
      tc_fence_after();
      // O / l for output columns [64 half, 64 half + 64) -> out[b, qpos, h*128 ..];
      // staged through this warp's 4 KB of the (idle) P buffer (128-byte rows,
      // 16-byte chunks XOR-swizzled by row), then 8 lanes per row
      const float inv = 1.f / l_sum;
      uint8_t* stage = sP + (warp - 2) * 32 * 128;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld32_sync(tmem + lane_base + kColO + 64 * half + c * 32, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int chunk = c * 4 + i;
          *reinterpret_cast<uint4*>(stage + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
              make_uint4(pack2<T16>(v[8 * i] * inv, v[8 * i + 1] * inv),
                         pack2<T16>(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                         pack2<T16>(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                         pack2<T16>(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        }
      }
      __syncwarp();
      T16* out = static_cast<T16*>(a.o);
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int r = it * 4 + lane / 8, cc = lane % 8;
        const int t = qt * kBq + quarter * 32 + r;
        if (t < a.T)
          *reinterpret_cast<uint4*>(out + ((int64_t)b * a.T + t) * (a.H * kHd) + h * kHd +
                                    64 * half + cc * 8) =
              *reinterpret_cast<const uint4*>(stage + r * 128 + ((cc ^ (r & 7)) << 4));
      }
    } else {
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// [outer..., T, 128] 16-bit rows: dims (128, T, d2[, d3]) with the given byte
// strides of dims 2 and 3; boxes of 64 columns x 128 rows. Rows >= T read as 0.
bool make_rows_map(CUtensorMap* map, const void* base, bool half, int rank, uint64_t T,
                   uint64_t d2, uint64_t stride2, uint64_t d3, uint64_t stride3) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {128, T, d2, d3};
  cuuint64_t strides[3] = {256, stride2, stride3};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
            (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Status word of calls made without a model (bounded-wait timeouts).
__device__ uint32_t g_attn_status;

// The two-query-tile kernel (attn_tc2.cu) when NC_ATTN_V2=1 (measurement).
bool use_attn_v2() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("NC_ATTN_V2");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

}  // namespace

// q [B, H, T, 128]; K/V of layer `layer` at k + layer * layer_stride elements,
// each [B_cache, Hkv, t_max, 128] (only sequences 0..B-1 and rows < T used).
nc_status tc_attention_prefill_tc(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int T, int t_max, int n_layers,
                                  int64_t layer_stride, int layer, nc_dtype dt, uint32_t* status,
                                  cudaStream_t s) {
  const bool half = dt == NC_F16;
  CUtensorMap mq, mk, mv;
  const uint64_t kv_rows_bytes = (uint64_t)t_max * 256;
  if (!make_rows_map(&mq, q, half, 3, T, (uint64_t)B * H, (uint64_t)T * 256, 1, 0) ||
      !make_rows_map(&mk, k, half, 4, T, (uint64_t)B * Hkv, kv_rows_bytes, n_layers,
                     (uint64_t)layer_stride * 2) ||
      !make_rows_map(&mv, v, half, 4, T, (uint64_t)B * Hkv, kv_rows_bytes, n_layers,
                     (uint64_t)layer_stride * 2))
    return NC_ERR_CUDA;
  if (use_attn_v2()) {
    if (!status && cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_attn_status) != cudaSuccess)
      return NC_ERR_CUDA;
    // the two-tile kernel reads K/V of one layer (layer coordinate 0)
    if (n_layers == 1) return attn2_launch(mq, mk, mv, o, B, H, Hkv, T, half, status, s);
  }
  AttnArgs a;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.T = T;
  a.n_qt = (T + kBq - 1) / kBq;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kHd));
  a.o = o;
  if (!status && cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_attn_status) != cudaSuccess)
    return NC_ERR_CUDA;
  a.status = status;
  const unsigned grid = (unsigned)(a.n_qt * B * H);
  if (half) {
    static bool cfg = false;
    if (!cfg) {
      if (cudaFuncSetAttribute(attn_prefill_tc_kernel<f16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return NC_ERR_CUDA;
      cfg = true;
    }
    attn_prefill_tc_kernel<f16><<<grid, 320, kSmem, s>>>(mq, mk, mv, a, layer);
  } else {
    static bool cfg = false;
    if (!cfg) {
      if (cudaFuncSetAttribute(attn_prefill_tc_kernel<bf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return NC_ERR_CUDA;
      cfg = true;
    }
    attn_prefill_tc_kernel<bf16><<<grid, 320, kSmem, s>>>(mq, mk, mv, a, layer);
  }
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace nc
