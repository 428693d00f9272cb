// Causal flash attention for prefill on tcgen05 (head_dim 128, 16-bit Q/K/V,
// fp32 softmax and accumulation in TMEM), with grouped-query head sharing.
//
// Persistent: one CTA per SM walks a static list of work items (128 queries of
// one (sequence, query head)), heaviest query tiles first, dealt to the CTAs
// in snake order (round r gives item r*G + c to CTA c, or r*G + G-1-c on odd
// rounds), which evens out the causal triangle. 352 threads:
//   warp 0      TMA: per item the Q tile, then K tiles of 128 keys into a
//               two-slot ring and V tiles into a three-slot ring, issued in the
//               order K0 K1, then V_j K_j+2 (keys at or past T read as zeros)
//   warp 1      TMEM owner; one thread issues S = Q K^T (M = N = K = 128) into
//               one of three TMEM score buffers, once P V of the buffer's
//               previous tile is done
//   warp 10     one thread issues O += P V with P read from TMEM (the A operand
//               of tcgen05.mma may live in tensor memory) and V an MN-major
//               shared-memory operand. Issuing eight MMAs blocks the issuing
//               thread for about as long as they execute, so two issuers keep
//               the tensor pipe fed where one would leave it idle while it waits
//   warps 2..9  softmax: warps w and w + 4 share the TMEM lane quarter w % 4
//               (thread = query row) and split the row's 128 key columns in two
//               halves; the pair exchanges row maxima through shared memory.
//               A thread masks keys past the query on the diagonal tile,
//               exponentiates in the log2 domain and writes its half of the
//               16-bit P row over the score columns it has read.
// The running max used as the exponent's reference is only raised when a row's
// max grows by more than 8 (log2 units): then that row of O is rescaled in TMEM
// (after the previous P V is complete). Otherwise p <= 2^8 and the reference
// stays, so the softmax of tile j never waits for the matrix products of tile
// j-1; the final O / l is the same either way. With three score buffers the
// tensor cores compute the scores of the next tiles, and those of the next
// item, while the softmax runs.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "tc.h"

namespace nc {

namespace {

constexpr int kHd = 128;
constexpr int kBq = 128;            // queries per item
constexpr int kBk = 128;            // keys per tile
constexpr int kTile = 128 * 128 * 2;   // 32 KB: a 128 x 128 16-bit tile (two 64-column boxes)
constexpr int kHalf = kTile / 2;
constexpr int kKring = 2;           // K ring slots
constexpr int kVring = 3;           // V ring slots
constexpr int kThreads = 352;
constexpr int kSbuf = 3;            // TMEM score buffers

// shared memory: Q | K ring[2] | V ring[3] | barriers | row-max exchange | row-sum exchange
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;
constexpr int kOffV = (1 + kKring) * kTile;
constexpr int kOffBar = (1 + kKring + kVring) * kTile;
constexpr int kOffX = kOffBar + 512;          // [2 parity][128 rows][2 halves] row maxima
constexpr int kOffL = kOffX + 2048;           // [128 rows][2 halves] final row sums
constexpr int kOffF = kOffL + 1024;           // [8 softmax warps] row-max flags (tile count)
constexpr size_t kSmem = kOffF + 64 + 1024;   // + alignment slack of the base

// TMEM columns: S/P buffers 0..383 (128 each), O 384..511
constexpr uint32_t kColO = kSbuf * 128, kTmemCols = 512;

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

// D(tmem) (+)= A(tmem) B(smem), 16-bit inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16kind_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32_sync(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// Shared-memory word with release / acquire semantics at CTA scope.
__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Waits until *flag >= target (a counter another warp of the CTA raises).
// Bounded like every other wait: sets ST_TIMEOUT and returns false after kWaitLimitNs.
__device__ __forceinline__ bool flag_wait(const uint32_t* flag, uint32_t target, uint32_t* status) {
  if (ld_acquire_cta(flag) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    // back off between polls: the partner warp shares this SM sub-partition
    for (int i = 0; i < 32; ++i) {
      __nanosleep(20);
      if (ld_acquire_cta(flag) >= target) return true;
    }
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, ST_TIMEOUT);
      return false;
    }
  }
}

struct AttnArgs {
  int B, H, Hkv, T, n_qt, n_items;
  int pos0;           // absolute position of query row 0 (keys 0 .. pos0 + T - 1)
  float scale_log2;
  void* o;            // [B, T, H*128]
  uint32_t* status;
};

// Key tiles query tile qt reads: those holding keys up to its last query's position.
__device__ __forceinline__ int key_tiles(const AttnArgs& a, int qt) {
  return (a.pos0 + min(a.T, (qt + 1) * kBq) - 1) / kBk + 1;
}

// k-th item of CTA c (snake order over items sorted heaviest first), or -1
__device__ __forceinline__ int item_of(int k, int c, int G, int n_items) {
  const int it = k * G + ((k & 1) ? G - 1 - c : c);
  return it < n_items ? it : -1;
}

// Position i in a ring of N slots (a running count over the CTA's items) ->
// slot and phase parity.
template <int N>
struct RingPos {
  uint32_t i = 0;
  __device__ __forceinline__ int slot() const { return (int)(i % N); }
  __device__ __forceinline__ uint32_t par() const { return (i / N) & 1u; }
};

template <class T16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const AttnArgs a, int layer) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;          // 1: Q tile landed (tx)
  uint64_t* q_empty = bars + 1;     // 1: the item's last S is done (commit)
  uint64_t* k_full = bars + 2;      // 2: K slot landed (tx)
  uint64_t* k_empty = bars + 4;     // 2: K slot consumed (commit)
  uint64_t* v_full = bars + 6;      // 3: V slot landed (tx)
  uint64_t* v_empty = bars + 9;     // 3: V slot consumed (commit)
  uint64_t* s_full = bars + 12;     // 3: scores in TMEM buffer (commit)
  // 3: P of the tile in TMEM buffer b (8 softmax warps). One barrier per buffer:
  // the softmax may run up to three tiles ahead of the P V issue, and a phase
  // of buffer b cannot complete again before P V of its tile has been issued.
  uint64_t* p_full = bars + 15;
  // 3: P V of the tile in buffer b done (commit). Phase x of buffer b is the
  // tile 3x + b. Every wait on it is for a phase whose predecessor has already
  // been observed by the S issuer (before it issued the S that reused the
  // buffer), as parity waits require.
  uint64_t* o_done = bars + 18;
  uint64_t* o_free = bars + 21;     // 1: the item's O has been read out (8 softmax warps)
  // [quarter][3]: the two softmax warps of a lane quarter exchange the final row
  // sums through slot 2 (2 arrivals; slots 0 and 1 unused)
  uint64_t* xbar = bars + 22;       // 12
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 34);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 35);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = gridDim.x, c = blockIdx.x;
  const int per_qt = a.B * a.H;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kKring; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVring; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < kSbuf; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(o_free, 8);
    for (int i = 0; i < 12; ++i) mbar_init(&xbar[i], 2);
    *abort_flag = 0;
    for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t*>(smem + kOffF)[i] = 0u;
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
      RingPos<kKring> kp;
      RingPos<kVring> vp;
      bool ok = true;
      int n_items_here = 0;
      auto load_k = [&](int j, int bg) -> bool {
        if (!mbar_wait_sleep(&k_empty[kp.slot()], kp.par() ^ 1u, a.status)) return false;
        uint8_t* d = smem + kOffK + kp.slot() * kTile;
        mbar_arrive_expect_tx(&k_full[kp.slot()], kTile);
        tma_load_4d(d, &tmK, &k_full[kp.slot()], 0, j * kBk, bg, layer);
        tma_load_4d(d + kHalf, &tmK, &k_full[kp.slot()], 64, j * kBk, bg, layer);
        ++kp.i;
        return true;
      };
      auto load_v = [&](int j, int bg) -> bool {
        if (!mbar_wait_sleep(&v_empty[vp.slot()], vp.par() ^ 1u, a.status)) return false;
        uint8_t* d = smem + kOffV + vp.slot() * kTile;
        mbar_arrive_expect_tx(&v_full[vp.slot()], kTile);
        tma_load_4d(d, &tmV, &v_full[vp.slot()], 0, j * kBk, bg, layer);
        tma_load_4d(d + kHalf, &tmV, &v_full[vp.slot()], 64, j * kBk, bg, layer);
        ++vp.i;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int item = item_of(k, c, G, a.n_items);
        if (item < 0 || *abort_flag) break;
        const int qt = a.n_qt - 1 - item / per_qt, bh = item % per_qt;
        const int bg = (bh / a.H) * a.Hkv + (bh % a.H) / (a.H / a.Hkv);
        const int n = key_tiles(a, qt);
        // Q of the previous item is no longer read once its last S is done
        if (k > 0 && !mbar_wait_sleep(q_empty, (k - 1) & 1, a.status)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, kTile);
        tma_load_3d(smem + kOffQ, &tmQ, q_full, 0, qt * kBq, bh);
        tma_load_3d(smem + kOffQ + kHalf, &tmQ, q_full, 64, qt * kBq, bh);
        ++n_items_here;
        // K_j+2 after V_j: the K ring frees a slot when S_j is done, the V ring
        // when P V_j-3 is done; neither wait can depend on a later load
        for (int j = 0; j < n && j < kKring && ok; ++j) ok = load_k(j, bg);
        for (int j = 0; j < n && ok; ++j) {
          ok = load_v(j, bg);
          if (ok && j + kKring < n) ok = load_k(j + kKring, bg);
        }
      }
      if (!ok) *abort_flag = 1;
      // copies in flight must land before shared memory is released
      if (n_items_here > 0) mbar_wait_sleep(q_full, (n_items_here - 1) & 1, a.status);
      for (uint32_t i = kp.i > kKring ? kp.i - kKring : 0; i < kp.i; ++i)
        mbar_wait_sleep(&k_full[i % kKring], (i / kKring) & 1u, a.status);
      for (uint32_t i = vp.i > kVring ? vp.i - kVring : 0; i < vp.i; ++i)
        mbar_wait_sleep(&v_full[i % kVring], (i / kVring) & 1u, a.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- S issuer
      constexpr uint32_t kIdS = idesc_f32acc(Fmt16<T16>::code, 128, 128);
      const uint32_t sQ = smem_u32(smem + kOffQ);
      RingPos<kKring> kp;
      uint32_t g = 0;   // running tile count over the CTA's items
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int item = item_of(k, c, G, a.n_items);
        if (item < 0 || *abort_flag) break;
        const int n = key_tiles(a, a.n_qt - 1 - item / per_qt);
        if (!mbar_wait_sleep(q_full, k & 1, a.status)) { ok = false; break; }
        for (int j = 0; j < n; ++j) {
          const uint32_t gg = g + j;
          // the buffer's previous user is P V of tile gg - 3 (phase (gg-3)/3 of
          // its barrier; this thread waits on every phase of it in order)
          if ((gg >= kSbuf &&
               !mbar_wait_sleep(&o_done[gg % kSbuf], ((gg - kSbuf) / kSbuf) & 1u, a.status)) ||
              !mbar_wait_sleep(&k_full[kp.slot()], kp.par(), a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + kOffK + kp.slot() * kTile);
          const uint32_t d = tmem + (gg % kSbuf) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t da = sdesc_kmajor_sw128(sQ + (kk >> 2) * kHalf + (kk & 3) * 32);
            const uint64_t db = sdesc_kmajor_sw128(sK + (kk >> 2) * kHalf + (kk & 3) * 32);
            mma_f16kind_ss(d, da, db, kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[gg % kSbuf]);
          mma_commit(&k_empty[kp.slot()]);
          ++kp.i;
        }
        if (!ok) break;
        mma_commit(q_empty);
        g += n;
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 10) {
    if (lane == 0) {
      // ---------------------------------------------------------- P V issuer
      constexpr uint32_t kIdO = idesc_f32acc(Fmt16<T16>::code, 128, 128) | (1u << 16);  // B MN-major
      RingPos<kVring> vp;
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int item = item_of(k, c, G, a.n_items);
        if (item < 0 || *abort_flag) break;
        const int n = key_tiles(a, a.n_qt - 1 - item / per_qt);
        for (int j = 0; j < n; ++j) {
          const uint32_t gg = g + j;
          // P of the tile in TMEM; the first product of an item overwrites O, so
          // the previous item's O must have been read out
          if (!mbar_wait_sleep(&p_full[gg % kSbuf], (gg / kSbuf) & 1u, a.status) ||
              (j == 0 && k > 0 && !mbar_wait_sleep(o_free, (k - 1) & 1, a.status)) ||
              !mbar_wait_sleep(&v_full[vp.slot()], vp.par(), a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O (+)= P V: P of keys 16kk..16kk+15 at TMEM columns 8kk (+32 for the
          // second half of the keys, written by the other softmax warp)
          const uint32_t sV = smem_u32(smem + kOffV + vp.slot() * kTile);
          const uint32_t pa = tmem + (gg % kSbuf) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t db = sdesc_mnmajor_sw128(sV + kk * 16 * 128, kHalf);
            mma_f16kind_ts(tmem + kColO, pa + kk * 8 + (kk >= 4 ? 32 : 0), db, kIdO,
                           (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&o_done[gg % kSbuf]);
          mma_commit(&v_empty[vp.slot()]);
          ++vp.i;
        }
        g += n;
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------- softmax (2..9)
    const int quarter = warp % 4;
    const int half = (warp - 2) / 4;          // key / output columns [64 half, 64 half + 64)
    const int row = quarter * 32 + lane;      // query row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + kOffX);
    float* xl = reinterpret_cast<float*>(smem + kOffL);
    uint64_t* qbar = xbar + 3 * quarter;      // this quarter's exchange barriers
    // row-max flags: warp w publishes the count of tiles whose maxima it has
    // written; its partner (same lane quarter, other half) is warp w +- 4
    uint32_t* flags = reinterpret_cast<uint32_t*>(smem + kOffF);
    uint32_t* my_flag = flags + (warp - 2);
    const uint32_t* partner_flag = flags + ((warp - 2) ^ 4);
    T16* out = static_cast<T16*>(a.o);
    uint32_t g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = item_of(k, c, G, a.n_items);
      if (item < 0 || *abort_flag) break;
      const int qt = a.n_qt - 1 - item / per_qt, bh = item % per_qt;
      const int b = bh / a.H, h = bh % a.H;
      const int n = key_tiles(a, qt);
      const int qrow = qt * kBq + row;     // row of q and of the output
      const int qpos = a.pos0 + qrow;      // its absolute position
      // tiles from this one on hold keys past the tile's first query: masked
      const int first_masked = (a.pos0 + qt * kBq) / kBk;
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int j = 0; j < n; ++j) {
        const uint32_t gg = g + j;
        const uint32_t sb = tmem + lane_base + (gg % kSbuf) * 128 + 64 * half;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[gg % kSbuf], (gg / kSbuf) & 1u, a.status));
        if (!ok) break;
        tc_fence_after();
        // this half of the score row in one 64-column TMEM load; causal mask
        float sv[64];
        tmem_ld64_sync(sb, sv);
        if (j >= first_masked) {
          const int kmax = qpos - j * kBk - 64 * half;   // keys i > kmax are masked
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > kmax) sv[i] = -INFINITY;
        }
        // row max over both halves (raw scores; the scale > 0 is applied to the max
        // and folded into the exponent's FMA), exchanged through shared memory
        // (a tree: eight independent partial maxima, then three levels)
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = sv[u];
#pragma unroll
        for (int i = 8; i < 64; ++i) m8[i & 7] = fmaxf(m8[i & 7], sv[i]);
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int u = 0; u < w; ++u) m8[u] = fmaxf(m8[u], m8[u + w]);
        float mx = m8[0];
        const int xp = gg & 1;
        xch[(xp * 128 + row) * 2 + half] = mx;
        __syncwarp();
        if (lane == 0) st_release_cta(my_flag, gg + 1);
        ok = __all_sync(0xffffffffu, flag_wait(partner_flag, gg + 1, a.status));
        if (!ok) break;
        mx = fmaxf(mx, xch[(xp * 128 + row) * 2 + (half ^ 1)]) * a.scale_log2;
        // raise the reference only when the max outgrows it by 2^8
        const bool raise = mx > m_ref + 8.f;
        const float m_new = raise ? mx : m_ref;
        const float corr = raise ? ex2_approx(m_ref - m_new) : 1.f;   // 0 on the first tile
        // p = 2^(s - m) packed to 16 bits, this half's row sum (four partial sums)
        float ps4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2_approx(fmaf(sv[2 * i], a.scale_log2, -m_new));
          const float p1 = ex2_approx(fmaf(sv[2 * i + 1], a.scale_log2, -m_new));
          ps4[i & 3] += p0 + p1;
          pk[i] = pack2<T16>(p0, p1);
        }
        const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        l_sum = l_sum * corr + psum;
        m_ref = m_new;
        // a raised reference rescales this half of the O row, after P V of the
        // previous tile is complete (the first tile of an item overwrites O)
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          ok = __all_sync(0xffffffffu, mbar_wait(&o_done[(gg - 1) % kSbuf],
                                                 ((gg - 1) / kSbuf) & 1u, a.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            float v[32];
            uint32_t w[32];
            const uint32_t oc = tmem + lane_base + kColO + 64 * half + cc * 32;
            tmem_ld32_sync(oc, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * corr);
            tmem_st32_sync(oc, w);
          }
        }
        // P over the first 32 columns of this half's (already read) scores
        tmem_st32_sync(sb, pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[gg % kSbuf]);
      }
      if (!ok) break;
      const uint32_t glast = g + n - 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&o_done[glast % kSbuf], (glast / kSbuf) & 1u, a.status));
      if (!ok) break;
      // the row sum is the two halves' sums (same reference max)
      xl[row * 2 + half] = l_sum;
      __syncwarp();
      if (lane == 0) mbar_arrive(&qbar[2]);
      ok = __all_sync(0xffffffffu, mbar_wait(&qbar[2], k & 1, a.status));
      if (!ok) break;
      l_sum += xl[row * 2 + (half ^ 1)];
      tc_fence_after();
      // O / l for output columns [64 half, 64 half + 64) -> out[b, qrow, h*128 ..]
      const float inv = 1.f / l_sum;
      const bool valid = qrow < a.T;
      T16* orow = out + ((int64_t)b * a.T + (valid ? qrow : 0)) * (a.H * kHd) + h * kHd + 64 * half;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
        tmem_ld32_sync(tmem + lane_base + kColO + 64 * half + cc * 32, v);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(orow + cc * 32 + 8 * i) =
                make_uint4(pack2<T16>(v[8 * i] * inv, v[8 * i + 1] * inv),
                           pack2<T16>(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                           pack2<T16>(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                           pack2<T16>(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      g += n;
    }
    if (!ok) *abort_flag = 1;
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

}  // namespace

// q [B, H, T, 128]; K/V of layer `layer` at k + layer * layer_stride elements,
// each [B_cache, Hkv, t_max, 128] (only sequences 0..B-1 and rows < T used).
nc_status tc_attention_prefill_tc(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int T, int pos0, int t_max, int n_layers,
                                  int64_t layer_stride, int layer, nc_dtype dt, uint32_t* status,
                                  cudaStream_t s) {
  if (pos0 < 0 || pos0 + T > t_max) return NC_ERR_INVALID_ARG;
  const bool half = dt == NC_F16;
  CUtensorMap mq, mk, mv;
  const uint64_t kv_rows_bytes = (uint64_t)t_max * 256;
  const uint64_t n_keys = (uint64_t)pos0 + T;   // cache rows at or past it read as zeros
  if (!make_rows_map(&mq, q, half, 3, T, (uint64_t)B * H, (uint64_t)T * 256, 1, 0) ||
      !make_rows_map(&mk, k, half, 4, n_keys, (uint64_t)B * Hkv, kv_rows_bytes, n_layers,
                     (uint64_t)layer_stride * 2) ||
      !make_rows_map(&mv, v, half, 4, n_keys, (uint64_t)B * Hkv, kv_rows_bytes, n_layers,
                     (uint64_t)layer_stride * 2))
    return NC_ERR_CUDA;
  AttnArgs a;
  a.pos0 = pos0;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.T = T;
  a.n_qt = (T + kBq - 1) / kBq;
  a.n_items = a.n_qt * B * H;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kHd));
  a.o = o;
  if (!status && cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_attn_status) != cudaSuccess)
    return NC_ERR_CUDA;
  a.status = status;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NC_ERR_CUDA;
  // one persistent CTA per SM (at most one per item)
  const unsigned grid = (unsigned)std::min(a.n_items, sms);
  if (half) {
    if (!ensure_dyn_smem((const void*)attn_prefill_tc_kernel<f16>, kSmem)) return NC_ERR_CUDA;
    attn_prefill_tc_kernel<f16><<<grid, kThreads, kSmem, s>>>(mq, mk, mv, a, layer);
  } else {
    if (!ensure_dyn_smem((const void*)attn_prefill_tc_kernel<bf16>, kSmem)) return NC_ERR_CUDA;
    attn_prefill_tc_kernel<bf16><<<grid, kThreads, kSmem, s>>>(mq, mk, mv, a, layer);
  }
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace nc
