// One decode step of the whole model in one persistent launch (16-bit path,
// head_dim 128, up to 32 sequences per launch).
//
// Decode is bound by HBM: every step streams all projection weights and every
// cached K/V row once, and each of them is used by only B <= 32 tokens. With one
// kernel per projection the step pays a launch, a ramp and a tail per kernel
// (about 180 of them for a 20-layer model), which costs more than the streaming
// itself. Here one CTA per SM runs the whole step:
//
//   warp 0 (producer)   one thread streams the CTA's share of every weight
//                       matrix (packed in mma-fragment order, 8 KB units, 1-D
//                       bulk copies) and of the KV cache (2-D TMA tiles of 16
//                       positions, 128-byte swizzle) into a ring of 8 KB stages.
//                       Nothing it loads depends on the step's activations, so
//                       it runs ahead across the grid barriers of the phases.
//   warps 1..8          consume the ring phase by phase, separated by grid
//                       barriers:
//     P0       embedding x = wte[token]; zero the accumulators of the step
//     per layer:
//       QKV    acc = x Wqkv^T (x un-normalised: RMSNorm has no gain, so the
//              norm is one scale per token, applied after the barrier); the CTAs
//              that cover feature group 0 also sum x^2 for that scale
//       ATTN   RoPE + QK norm of q and of the new k, cache write of the new
//              k / v, split-KV attention over positions 0..pos (all query heads
//              of a KV head share one pass over K/V); the last CTA of each
//              (sequence, KV head) merges the partial softmax states
//       O      x += att Wo^T
//       FC     hacc = x Wfc^T (un-normalised, sum of x^2 as in QKV)
//       PROJ   x += relu(r hacc)^2 Wproj^T
//     FNORM    xn = RMSNorm(x) in mma-fragment order
//     LM       logits = xn Wlm^T
//     ARGMAX   greedy token per sequence (lowest index on ties)
//
// GEMV phases: the weight matrix [N, K] is cut into units of 128 rows x 32
// columns (8 KB). Units are ordered row-group-major and each CTA takes an equal
// contiguous range of them, so every CTA streams the same number of bytes. Warp
// w owns the 16 rows w*16.. of the unit (mma.sync m16n8k16: the weights are the
// A operand, the tokens the 8-wide N tiles); at the end of a row group's run the
// warp adds its 16 x B partial sums into the fp32 output with vector reductions.
// Projection outputs therefore sum in a run-dependent order (fp32).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "nc_internal.h"
#include "decode_fused.h"

namespace nc {
namespace dec {

constexpr int kCons = 8;                   // consumer warps
constexpr int kThreads = 32 * (kCons + 1);
constexpr int kStage = 8192;               // bytes of one ring stage
constexpr int kUnitRows = 128;             // weight rows of one unit (8 warps x 16)
constexpr int kUnitCols = 32;              // weight columns of one unit (two k16 steps)
constexpr int kHd = 128;
constexpr int kMergeStride = 132;          // floats per row of a warp's merge area
constexpr int kMergeBytes = kCons * (16 * kMergeStride + 32) * 4;
constexpr int kXposeBytes = kCons * 16 * 33 * 4;

enum Phase : int { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_FC = 3, PH_PROJ = 4 };
enum ActKind : int { ACT_X32 = 0, ACT_A16 = 1, ACT_H32 = 2, ACT_FRAG = 3 };

// ---------------------------------------------------------------- primitives
__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

template <class T16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<f16>(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<bf16>(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of element column-chunk c16 (16 bytes = 8 values) of row r in a
// [16 rows x 128 values] tile stored as two 64-column halves of 2 KB with the
// TMA 128-byte swizzle (chunk index XOR row % 8 inside each 1 KB block).
__device__ __forceinline__ uint32_t sw_off(int r, int c16) {
  return (uint32_t)((c16 >> 3) * 2048 + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------ work ranges
// Contiguous share [lo, hi) of `total` items for CTA c of P. With fewer items
// than CTAs, CTA c < total takes item c; otherwise every share is non-empty. So
// the CTAs that touch any run of consecutive items are consecutive themselves.
__host__ __device__ __forceinline__ void share(int64_t total, int c, int P, int64_t& lo,
                                               int64_t& hi) {
  if (total < P) {
    lo = c < total ? c : total;
    hi = c + 1 < total ? c + 1 : total;
  } else {
    lo = total * c / P;
    hi = total * (c + 1) / P;
  }
}
// The CTA whose share contains item f.
__host__ __device__ __forceinline__ int owner_of(int64_t total, int64_t f, int P) {
  return total < P ? (int)f : (int)(((f + 1) * P - 1) / total);
}

// Attention work: tiles of 16 positions over (sequence, KV head) pairs bg. With no
// more pairs than CTAs, every pair gets its own consecutive block of
// floor or ceil(P / pairs) CTAs and each CTA one contiguous tile range of one pair
// (one partial state per CTA); otherwise the flattened (pair, tile) space is
// shared evenly. attn_work gives CTA c's flattened range [f0, f1) (f = bg * T16 +
// tile); attn_group the CTAs holding tiles of pair bg: c_first, c_first + 1, ...
// (ns of them).
__host__ __device__ __forceinline__ void attn_work(int bhkv, int T16, int c, int P, int64_t& f0,
                                                   int64_t& f1) {
  if (bhkv <= P) {
    const int bg = (int)(((int64_t)(c + 1) * bhkv - 1) / P);
    const int cs = (int)((int64_t)bg * P / bhkv), ce = (int)((int64_t)(bg + 1) * P / bhkv);
    int64_t j0, j1;
    share(T16, c - cs, ce - cs, j0, j1);
    f0 = (int64_t)bg * T16 + j0;
    f1 = (int64_t)bg * T16 + j1;
  } else {
    share((int64_t)bhkv * T16, c, P, f0, f1);
  }
}
__host__ __device__ __forceinline__ void attn_group(int bhkv, int T16, int bg, int P, int& c_first,
                                                    int& ns) {
  if (bhkv <= P) {
    c_first = (int)((int64_t)bg * P / bhkv);
    const int n = (int)((int64_t)(bg + 1) * P / bhkv) - c_first;
    ns = n < T16 ? n : T16;
  } else {
    const int64_t total = (int64_t)bhkv * T16;
    c_first = owner_of(total, (int64_t)bg * T16, P);
    ns = owner_of(total, (int64_t)bg * T16 + T16 - 1, P) - c_first + 1;
  }
}

// ------------------------------------------------------------------- state
struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int n;
  int stage;
  uint32_t parity;
  __device__ __forceinline__ void advance() {
    if (++stage == n) {
      stage = 0;
      parity ^= 1u;
    }
  }
};

struct Shared {
  Ring ring;
  uint8_t* act;        // activation fragments / attention merge area
  int act_ksteps;      // capacity in k16 steps
  float* xpose;        // per-warp 16 x 32 transpose tiles
  uint8_t* sq;         // Q tile (16 x 128, swizzled)
  uint16_t* kvnew;     // new K row, new V row (16-bit)
  float* ss_s;         // [kMaxTok] per-token partial sums of squares
  volatile int* flag;  // [0] abort seen, [1] last-arriver flag, [2] barrier ok
};

__device__ __forceinline__ bool aborted(const Params& p) {
  return *reinterpret_cast<volatile uint32_t*>(p.abort) != 0;
}
__device__ __forceinline__ void raise_abort(const Params& p) {
  atomicOr(p.status, ST_TIMEOUT);
  atomicExch(p.abort, 1u);
}

// Trace mark m (0..3) of the phase that ends at grid barrier k: CTA 0, first
// consumer thread, only while a trace buffer is set.
__device__ __forceinline__ void trace_mark(const Params& p, int k, int m) {
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 32)
    p.trace[2 * p.nbar + 2 + 6 * (k - 1) + m] = global_timer_ns();
}

// Producer mark: when CTA 0's producer starts issuing the loads of the phase
// that ends at grid barrier k.
__device__ __forceinline__ void trace_producer(const Params& p, int k) {
  if (p.trace && blockIdx.x == 0) p.trace[2 * p.nbar + 2 + 6 * (k - 1) + 4] = global_timer_ns();
}

// Bounded wait on a ring barrier; false on timeout or abort.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, const Params& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (aborted(p)) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_abort(p);
      return false;
    }
  }
}

// Grid barrier number k (1-based) of this launch among the consumer warps of all
// CTAs. Returns false if the step was aborted.
__device__ bool grid_barrier(const Params& p, const Shared& sh, int k) {
  bar_consumers();
  const int tid = threadIdx.x - 32;
  if (tid == 0) {
    bool ok = true;
    const bool tr = p.trace && blockIdx.x == 0;
    if (tr) p.trace[2 * k - 1] = global_timer_ns();
    // release at GPU scope: this CTA's writes (ordered before this thread by the
    // CTA barrier above) are visible to any CTA that acquires the count
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p.bar_counter) : "memory");
    const unsigned long long target = p.bar_base + (unsigned long long)k * gridDim.x;
    uint64_t t0 = 0;
    int it = 0;
    while (ld_acquire_u64(p.bar_counter) < target) {
      if (++it == 32) {
        it = 0;
        if (aborted(p)) {
          ok = false;
          break;
        }
        const uint64_t t = global_timer_ns();
        if (t0 == 0) {
          t0 = t;
        } else if (t - t0 > kWaitLimitNs) {
          raise_abort(p);
          ok = false;
          break;
        }
      }
    }
    sh.flag[2] = ok ? 1 : 0;
    if (tr) p.trace[2 * k] = global_timer_ns();
  }
  bar_consumers();
  return sh.flag[2] != 0;
}

// --------------------------------------------------------- phase geometry
struct Gemv {
  const uint8_t* w;    // packed units
  int groups, kpairs;  // units = groups * kpairs
  float* out;          // fp32 [B, ldo]
  int ldo, n_valid;
  int act_kind;
  const void* act;     // source of the activations
  int act_ld;
  const float* ss_in;  // ACT_H32: sums of squares giving the per-token scale
  float* ss_out;       // ACT_X32: sums of squares of x accumulated here (or null)
};

__device__ __forceinline__ Gemv gemv_of(const Params& p, int l, int ph) {
  Gemv g{};
  const uint8_t* lw = p.wpack + (int64_t)l * p.layer_bytes;
  const int d = p.d, qd = p.H * kHd;
  switch (ph) {
    case PH_QKV:
      g.w = lw;
      g.groups = p.nqkv_pad / kUnitRows;
      g.kpairs = d / kUnitCols;
      g.out = p.qkv_acc + (int64_t)(l & 1) * kMaxTok * p.nqkv_pad;
      g.ldo = p.nqkv_pad;
      g.n_valid = p.nqkv;
      g.act_kind = ACT_X32;
      g.act = p.x;
      g.act_ld = d;
      g.ss_out = p.ss + (2 * l) * kMaxTok;
      break;
    case PH_O:
      g.w = lw + p.off_o;
      g.groups = d / kUnitRows;
      g.kpairs = qd / kUnitCols;
      g.out = p.x;
      g.ldo = d;
      g.n_valid = d;
      g.act_kind = ACT_A16;
      g.act = p.att;
      g.act_ld = qd;
      break;
    case PH_FC:
      g.w = lw + p.off_fc;
      g.groups = p.F / kUnitRows;
      g.kpairs = d / kUnitCols;
      g.out = p.hacc;
      g.ldo = p.F;
      g.n_valid = p.F;
      g.act_kind = ACT_X32;
      g.act = p.x;
      g.act_ld = d;
      g.ss_out = p.ss + (2 * l + 1) * kMaxTok;
      break;
    default:  // PH_PROJ
      g.w = lw + p.off_proj;
      g.groups = d / kUnitRows;
      g.kpairs = p.F / kUnitCols;
      g.out = p.x;
      g.ldo = d;
      g.n_valid = d;
      g.act_kind = ACT_H32;
      g.act = p.hacc;
      g.act_ld = p.F;
      g.ss_in = p.ss + (2 * l + 1) * kMaxTok;
      break;
  }
  return g;
}

__device__ __forceinline__ Gemv gemv_lm(const Params& p) {
  Gemv g{};
  g.w = p.wpack + (int64_t)p.L * p.layer_bytes;
  g.groups = p.vpad / kUnitRows;
  g.kpairs = p.d / kUnitCols;
  g.out = p.logits;
  g.ldo = p.V;
  g.n_valid = p.V;
  g.act_kind = ACT_FRAG;
  g.act = p.xnf;
  return g;
}

// Attention work: tiles of 16 positions over (sequence, KV head, tile).
__device__ __forceinline__ int attn_tiles(const Params& p) { return (p.pos + 1 + 15) / 16; }

// ================================================================ producer
__device__ void produce_gemv(const Params& p, Ring& r, const Gemv& g, uint64_t pol, bool& ok) {
  int64_t u0, u1;
  share((int64_t)g.groups * g.kpairs, blockIdx.x, gridDim.x, u0, u1);
  for (int64_t u = u0; u < u1 && ok; ++u) {
    if (!ring_wait(&r.empty[r.stage], r.parity ^ 1u, p)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&r.full[r.stage], kStage);
    bulk_load(r.base + (size_t)r.stage * kStage, g.w + u * kStage, kStage, &r.full[r.stage], pol);
    r.advance();
  }
}

__device__ void produce_attn(const Params& p, Ring& r, const CUtensorMap* tk, const CUtensorMap* tv,
                             int l, uint64_t pol, bool& ok) {
  const int T16 = attn_tiles(p);
  int64_t f0, f1;
  attn_work(p.B * p.Hkv, T16, blockIdx.x, gridDim.x, f0, f1);
  for (int64_t f = f0; f < f1 && ok; ++f) {
    const int j = (int)(f % T16);
    const int bg = (int)(f / T16);
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int64_t row = (((int64_t)l * p.cache_batch + p.b_off + b) * p.Hkv + g) * p.t_max + 16 * j;
    if (!ring_wait(&r.empty[r.stage], r.parity ^ 1u, p)) {
      ok = false;
      break;
    }
    uint8_t* dst = r.base + (size_t)r.stage * kStage;
    mbar_arrive_expect_tx(&r.full[r.stage], kStage);
    tma_load_2d_hint(dst, tk, &r.full[r.stage], 0, (int32_t)row, pol);
    tma_load_2d_hint(dst + 2048, tk, &r.full[r.stage], 64, (int32_t)row, pol);
    tma_load_2d_hint(dst + 4096, tv, &r.full[r.stage], 0, (int32_t)row, pol);
    tma_load_2d_hint(dst + 6144, tv, &r.full[r.stage], 64, (int32_t)row, pol);
    r.advance();
  }
}

__device__ void producer(const Params& p, Shared& sh, const CUtensorMap* tk, const CUtensorMap* tv) {
  Ring& r = sh.ring;
  const uint64_t pol = l2_policy_evict_first();
  bool ok = true;
  for (int l = 0; l < p.L && ok; ++l) {
    const int k = 2 + 5 * l;   // grid barrier that ends this layer's QKV phase
    trace_producer(p, k);
    produce_gemv(p, r, gemv_of(p, l, PH_QKV), pol, ok);
    trace_producer(p, k + 1);
    produce_attn(p, r, tk, tv, l, pol, ok);
    trace_producer(p, k + 2);
    produce_gemv(p, r, gemv_of(p, l, PH_O), pol, ok);
    trace_producer(p, k + 3);
    produce_gemv(p, r, gemv_of(p, l, PH_FC), pol, ok);
    trace_producer(p, k + 4);
    produce_gemv(p, r, gemv_of(p, l, PH_PROJ), pol, ok);
  }
  trace_producer(p, 5 * p.L + 3);
  if (ok) produce_gemv(p, r, gemv_lm(p), pol, ok);
  if (!ok) {
    // Let every copy already issued land before the CTA's shared memory goes
    // away: the latest fill of each stage completes its full barrier's phase.
    for (int i = 0; i < r.n; ++i) {
      r.stage = (r.stage + r.n - 1) % r.n;
      if (r.stage == r.n - 1) r.parity ^= 1u;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&r.full[r.stage], r.parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
}

// Asynchronous global -> shared copies of 4 or 8 bytes (cp.async, cached in L1 as
// well: the copies of one staging pass are all in flight at once and hold no
// registers). cp_async_wait_all makes this thread's copies visible to itself.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_all;\n" ::: "memory");
}

// =============================================================== consumers
// Stages activation k16 steps [ks0, ks1) of the current phase into shared
// memory as mma B fragments: entry ((ks - ks0) * NT + nt) * 32 + lane holds the
// two 32-bit registers of lane `lane` for tokens 8nt..8nt+7.
template <int NT, class T16>
__device__ void stage_act(const Params& p, const Shared& sh, const Gemv& g, int ks0, int ks1,
                          int ss_c0, int ss_c1, int ks0b = 0, int ks1b = 0) {
  // Entry i of the window holds lane (i % 32)'s B fragment of token tile
  // (i / 32) % NT. A thread handles entries tid, tid + 256, ...; as NT divides 8,
  // all of them belong to one token: tok = (warp % NT) * 8 + lane / 4. Each pass
  // issues all of a thread's loads before their first use (one L2 round trip).
  // For ACT_X32 the squares of the columns in [ss_c0, ss_c1) are summed in a
  // register and added to g.ss_out; for ACT_H32 the token's norm scale is read
  // once before the loads.
  constexpr int kBatch = 8;
  uint2* dst = reinterpret_cast<uint2*>(sh.act);
  const int tid = threadIdx.x - 32;
  const int lane = tid & 31;
  const int tok = ((tid >> 5) % NT) * 8 + (lane >> 2);
  const bool tok_ok = tok < p.B;
  // entries of k steps [ks0, ks1) come first, then those of [ks0b, ks1b)
  const int lenA = ks1 - ks0;
  const int n = (lenA + (ks1b - ks0b)) * NT * 32;
  auto ks_of = [&](int i) {
    const int e = (i >> 5) / NT;
    return e < lenA ? ks0 + e : ks0b + (e - lenA);
  };
  const bool want_ss = g.act_kind == ACT_X32 && g.ss_out && ss_c0 < ss_c1;
  // the token's norm scale (ACT_H32) is loaded here and used after the first
  // batch of loads is in flight
  const float ss_tok = (g.act_kind == ACT_H32 && tok_ok) ? __ldcg(g.ss_in + tok) : 0.f;
  float ssum = 0.f;
  // Asynchronous path, whenever the fp32 sources' landing zone (16 bytes per entry,
  // after the 8-byte fragments) fits in the activation area: every copy of the
  // pass is issued before the first is waited for (one L2 round trip, no
  // registers held). 16-bit sources are copied straight into their fragments.
  const bool f32src = g.act_kind == ACT_X32 || g.act_kind == ACT_H32;
  if ((int64_t)n * (f32src ? 24 : 8) <= p.act_bytes) {
    float4* land = reinterpret_cast<float4*>(sh.act + (size_t)n * 8);
    for (int i = tid; i < n; i += 256) {
      const int ks = ks_of(i);
      if (g.act_kind == ACT_FRAG) {
        cp_async8(dst + i, reinterpret_cast<const uint2*>(g.act) + ((int64_t)ks * NT + ((i >> 5) % NT)) * 32 + (i & 31));
        continue;
      }
      if (!tok_ok) continue;
      const int kc = ks * 16 + 2 * (lane & 3);
      if (g.act_kind == ACT_A16) {
        const T16* src = static_cast<const T16*>(g.act) + (int64_t)tok * g.act_ld + kc;
        uint32_t* d = reinterpret_cast<uint32_t*>(dst + i);
        cp_async4(d, src);
        cp_async4(d + 1, src + 8);
      } else {
        const float* src = static_cast<const float*>(g.act) + (int64_t)tok * g.act_ld + kc;
        float* d = reinterpret_cast<float*>(land + i);
        cp_async8(d, src);
        cp_async8(d + 2, src + 8);
      }
    }
    cp_async_wait_all();
    if (g.act_kind == ACT_FRAG) return;
    if (g.act_kind == ACT_A16) {
      if (!tok_ok)
        for (int i = tid; i < n; i += 256) dst[i] = make_uint2(0u, 0u);
      return;
    }
    const float rscale = rsqrtf(ss_tok / (float)p.d + p.eps);
    for (int i = tid; i < n; i += 256) {
      float4 x = tok_ok ? land[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      if (want_ss && (i >> 5) / NT < lenA) {   // columns of the first range only
        const int kc = ks_of(i) * 16 + 2 * (lane & 3);
        if (kc >= ss_c0 && kc < ss_c1) ssum += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      }
      if (g.act_kind == ACT_H32) {
        x.x = fmaxf(x.x * rscale, 0.f);
        x.y = fmaxf(x.y * rscale, 0.f);
        x.z = fmaxf(x.z * rscale, 0.f);
        x.w = fmaxf(x.w * rscale, 0.f);
        x = make_float4(x.x * x.x, x.y * x.y, x.z * x.z, x.w * x.w);
      }
      dst[i] = make_uint2(pack2<T16>(x.x, x.y), pack2<T16>(x.z, x.w));
    }
    if (want_ss) {
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      if ((lane & 3) == 0 && tok_ok && ssum != 0.f) atomicAdd(g.ss_out + tok, ssum);
    }
    return;
  }
  for (int i0 = tid; i0 < n; i0 += 256 * kBatch) {
    if (g.act_kind == ACT_FRAG) {
      const uint2* src = reinterpret_cast<const uint2*>(g.act);
      uint2 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * 256;
        if (i < n) v[u] = __ldcg(src + ((int64_t)ks_of(i) * NT + ((i >> 5) % NT)) * 32 + (i & 31));
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * 256;
        if (i < n) dst[i] = v[u];
      }
      continue;
    }
    if (g.act_kind == ACT_A16) {
      uint2 w[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * 256;
        const int kc = ks_of(i) * 16 + 2 * (lane & 3);
        w[u] = make_uint2(0u, 0u);
        if (i < n && tok_ok) {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(
              static_cast<const T16*>(g.act) + (int64_t)tok * g.act_ld + kc);
          w[u].x = __ldcg(src);
          w[u].y = __ldcg(src + 4);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (i0 + u * 256 < n) dst[i0 + u * 256] = w[u];
      continue;
    }
    float4 v[kBatch];   // x[tok, kc], x[tok, kc + 1], x[tok, kc + 8], x[tok, kc + 9]
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * 256;
      const int kc = ks_of(i) * 16 + 2 * (lane & 3);
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n && tok_ok) {
        const float* src = static_cast<const float*>(g.act) + (int64_t)tok * g.act_ld + kc;
        const float2 a = __ldcg(reinterpret_cast<const float2*>(src));
        const float2 b = __ldcg(reinterpret_cast<const float2*>(src + 8));
        v[u] = make_float4(a.x, a.y, b.x, b.y);
      }
    }
    const float rscale = rsqrtf(ss_tok / (float)p.d + p.eps);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * 256;
      if (i >= n) continue;
      float4 x = v[u];
      if (want_ss && (i >> 5) / NT < lenA) {   // columns of the first range only
        const int kc = ks_of(i) * 16 + 2 * (lane & 3);
        if (kc >= ss_c0 && kc < ss_c1) ssum += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      }
      if (g.act_kind == ACT_H32) {
        x.x = fmaxf(x.x * rscale, 0.f);
        x.y = fmaxf(x.y * rscale, 0.f);
        x.z = fmaxf(x.z * rscale, 0.f);
        x.w = fmaxf(x.w * rscale, 0.f);
        x = make_float4(x.x * x.x, x.y * x.y, x.z * x.z, x.w * x.w);
      }
      dst[i] = make_uint2(pack2<T16>(x.x, x.y), pack2<T16>(x.z, x.w));
    }
  }
  if (want_ss) {
    // the four lanes of a quad hold the same token
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
    if ((lane & 3) == 0 && tok_ok && ssum != 0.f) atomicAdd(g.ss_out + tok, ssum);
  }
}

// Adds the warp's 16 x (8 NT) partial sums into out[tok, row0 + 0..15].
template <int NT>
__device__ __forceinline__ void flush_rows(const Params& p, const Shared& sh, const Gemv& g,
                                           int row0, float (&acc)[NT][4]) {
  const int warp = threadIdx.x / 32 - 1, lane = threadIdx.x % 32;
  const int gq = lane >> 2, tq = lane & 3;
  float* t = sh.xpose + warp * 16 * 33;   // [16 rows][33] (row = feature)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // token columns 8nt + 2tq (+1); rows gq and gq + 8
    const int c = nt * 8 + 2 * tq;
    if (c < 32) {
      t[gq * 33 + c] = acc[nt][0];
      t[gq * 33 + c + 1] = acc[nt][1];
      t[(gq + 8) * 33 + c] = acc[nt][2];
      t[(gq + 8) * 33 + c + 1] = acc[nt][3];
    }
  }
  __syncwarp();
  // 4 quads of features x up to 32 tokens: lane handles token `lane`
  const int tok = lane;
  if (tok < p.B) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = row0 + 4 * q;
      if (f < g.n_valid) {
        float* dst = g.out + (int64_t)tok * g.ldo + f;
        red_add_v4(dst, t[(4 * q) * 33 + tok], t[(4 * q + 1) * 33 + tok], t[(4 * q + 2) * 33 + tok],
                   t[(4 * q + 3) * 33 + tok]);
      }
    }
  }
  __syncwarp();
}

template <int NT, class T16>
__device__ bool consume_gemv(const Params& p, Shared& sh, const Gemv& g, int k) {
  const int warp = threadIdx.x / 32 - 1, lane = threadIdx.x % 32;
  Ring& r = sh.ring;
  int64_t u0, u1;
  const int64_t units = (int64_t)g.groups * g.kpairs;
  share(units, blockIdx.x, gridDim.x, u0, u1);
  if (u0 >= u1) return true;
  // The sum of squares of x over the columns of row group 0 this CTA covers is
  // taken while staging that run (runs in row group 0 only start this CTA's range).
  int ss_c0 = 0, ss_c1 = 0;
  if (g.ss_out && u0 < g.kpairs) {
    ss_c0 = (int)u0 * kUnitCols;
    ss_c1 = (int)std::min<int64_t>(u1, g.kpairs) * kUnitCols;
  }
  // activation window [win0, win1) in k16 steps, staged on demand. A share of
  // exactly two runs (the end of one row group, the start of the next) that fits
  // is staged in one pass: run 1's k steps, then run 2's at offset `off2`.
  int win0 = 0, win1 = 0;
  int two_b0 = -1, two_off = 0;   // run 2's first k step and its offset, if both staged
  const int cap = sh.act_ksteps;
  {
    const int kpa = (int)(u0 % g.kpairs);
    const int64_t n1 = g.kpairs - kpa;   // units of run 1
    const int64_t n2 = (u1 - u0) - n1;   // units of run 2
    if (n1 > 0 && n2 > 0 && n2 <= g.kpairs && 2 * (n1 + n2) <= cap) {
      bar_consumers();
      trace_mark(p, k, 3);
      win0 = 2 * kpa;
      win1 = 2 * g.kpairs;
      two_b0 = 0;
      two_off = 2 * (int)n1;
      stage_act<NT, T16>(p, sh, g, win0, win1, ss_c0, ss_c1, 0, 2 * (int)n2);
      bar_consumers();
      trace_mark(p, k, 0);
    }
  }
  int64_t u = u0;
  while (u < u1) {
    const int grp = (int)(u / g.kpairs);
    const int kp0 = (int)(u % g.kpairs);
    const int kp1 = (int)std::min<int64_t>(g.kpairs, kp0 + (u1 - u));
    const bool second = two_b0 >= 0 && u > u0;   // run 2 of a two-run share
    if (!second && (2 * kp0 < win0 || 2 * kp1 > win1)) {
      // Every warp is done with the old window (all warps walk the same units).
      // A later row group needs the same columns again: stage the whole K once
      // if it fits, else this run's columns.
      bar_consumers();
      trace_mark(p, k, 3);
      if (u1 - u > g.kpairs && 2 * g.kpairs <= cap) {
        win0 = 0;
        win1 = 2 * g.kpairs;
      } else {
        win0 = 2 * kp0;
        win1 = std::min(2 * kp1, win0 + cap);
      }
      stage_act<NT, T16>(p, sh, g, win0, win1, ss_c0, ss_c1);
      bar_consumers();
      trace_mark(p, k, 0);
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    for (int kp = kp0; kp < kp1; ++kp) {
      const int ks = 2 * kp;
      if (!second && ks + 2 > win1) {   // run longer than the window: slide it
        bar_consumers();
        win0 = ks;
        win1 = std::min(2 * kp1, win0 + cap);
        stage_act<NT, T16>(p, sh, g, win0, win1, ss_c0, ss_c1);
        bar_consumers();
      }
      if (!ring_wait(&r.full[r.stage], r.parity, p)) return false;
      const uint8_t* st = r.base + (size_t)r.stage * kStage;
      const uint2* bf = reinterpret_cast<const uint2*>(sh.act);
      {
        const uint4 a0 = *reinterpret_cast<const uint4*>(st + warp * 512 + lane * 16);
        const uint4 a1 = *reinterpret_cast<const uint4*>(st + 4096 + warp * 512 + lane * 16);
        const int ksl = second ? two_off + ks - two_b0 : ks - win0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 b0 = bf[(ksl * NT + nt) * 32 + lane];
          const uint2 b1 = bf[((ksl + 1) * NT + nt) * 32 + lane];
          mma16816<T16>(acc[nt], a0.x, a0.y, a0.z, a0.w, b0.x, b0.y);
          mma16816<T16>(acc[nt], a1.x, a1.y, a1.z, a1.w, b1.x, b1.y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[r.stage]);
      r.advance();
    }
    trace_mark(p, k, 1);
    flush_rows<NT>(p, sh, g, grp * kUnitRows + warp * 16, acc);
    trace_mark(p, k, 2);
    if (grp == 0) ss_c0 = ss_c1 = 0;   // the columns are counted once
    u += kp1 - kp0;
  }
  return true;
}

// ---------------------------------------------------------------- attention
// q (or k) head of sequence b: a = r * acc; RMS-normalised over its 128 values,
// then rotated by +theta(pos, i) on pairs (i, i + 64). Lane holds i = lane + 32 j.
__device__ __forceinline__ void rope_norm(const Params& p, const float* src, float r, float (&o)[4]) {
  const int lane = threadIdx.x % 32;
  float a[4];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a[j] = __ldcg(src + lane + 32 * j) * r;
    s += a[j] * a[j];
  }
  s = warp_sum(s);
  const float rn = rsqrtf(s * (1.f / kHd) + p.eps);
  const float* cs = p.cos_tab + (int64_t)p.pos * (kHd / 2);
  const float* sn = p.sin_tab + (int64_t)p.pos * (kHd / 2);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = lane + 32 * j;
    const float c = cs[i], sv = sn[i];
    const float lo = a[j], hi = a[j + 2];
    o[j] = (lo * c - hi * sv) * rn;
    o[j + 2] = (lo * sv + hi * c) * rn;
  }
}

template <class T16>
__device__ __forceinline__ void st16(uint8_t* tile, int r, int col, float v) {
  *reinterpret_cast<T16*>(tile + sw_off(r, col >> 3) + (col & 7) * 2) = from_f32<T16>(v);
}

template <class T16>
__device__ bool consume_attn(const Params& p, Shared& sh, int l, int k) {
  const int warp = threadIdx.x / 32 - 1, lane = threadIdx.x % 32;
  const int tid = threadIdx.x - 32;
  const int gq = lane >> 2, tq = lane & 3;
  Ring& r = sh.ring;
  const int T16n = attn_tiles(p);
  int64_t f0, f1;
  attn_work(p.B * p.Hkv, T16n, blockIdx.x, gridDim.x, f0, f1);
  const int G = p.H / p.Hkv;
  const int qd = p.H * kHd, kvd = p.Hkv * kHd;
  const float* acc_l = p.qkv_acc + (int64_t)(l & 1) * kMaxTok * p.nqkv_pad;
  const float* ss_l = p.ss + (2 * l) * kMaxTok;
  const int len = p.pos + 1;
  const int last_tile = T16n - 1;
  const int rp = p.pos - 16 * last_tile;   // row of pos in the last tile
  int64_t f = f0;
  while (f < f1) {
    const int bg = (int)(f / T16n);
    const int j0 = (int)(f % T16n);
    const int j1 = (int)std::min<int64_t>(T16n, j0 + (f1 - f));
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const float ssb = __ldcg(ss_l + b);   // used after the q/k/v loads are issued
    const float* accb = acc_l + (int64_t)b * p.nqkv_pad;
    // ---- Q tile of the group's query heads (rows >= G zero) and, in the CTA that
    // holds position pos, the new k / v row. Warp w prepares query rows w and w + 8;
    // warps 0 and 1 also the new k and v. All loads are issued before any use.
    const bool has_last = j1 == T16n;
    {
      const int nrow = (has_last && warp < 2) ? 3 : 2;
      float av[3][4];
      const float* cs = p.cos_tab + (int64_t)p.pos * (kHd / 2);
      const float* sn = p.sin_tab + (int64_t)p.pos * (kHd / 2);
      float cv[2], sv[2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        cv[jj] = cs[lane + 32 * jj];
        sv[jj] = sn[lane + 32 * jj];
      }
#pragma unroll
      for (int rr = 0; rr < 3; ++rr) {
        const int hh = warp + 8 * rr;
        const float* src = nullptr;
        if (rr < 2 && hh < G) src = accb + (g * G + hh) * kHd;
        if (rr == 2 && nrow == 3) src = accb + qd + (warp == 0 ? g * kHd : kvd + g * kHd);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) av[rr][jj] = src ? __ldcg(src + lane + 32 * jj) : 0.f;
      }
      const float rb = rsqrtf(ssb / (float)p.d + p.eps);
#pragma unroll
      for (int rr = 0; rr < 3; ++rr)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) av[rr][jj] *= rb;
#pragma unroll
      for (int rr = 0; rr < 3; ++rr) {
        if (rr == 2 && nrow < 3) break;
        const bool is_v = rr == 2 && warp == 1;
        float o[4];
        if (is_v) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) o[jj] = av[rr][jj];
        } else {
          float sq = 0.f;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) sq += av[rr][jj] * av[rr][jj];
          sq = warp_sum(sq);
          const float rn = rsqrtf(sq * (1.f / kHd) + p.eps);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const float lo = av[rr][jj], hi = av[rr][jj + 2];
            o[jj] = (lo * cv[jj] - hi * sv[jj]) * rn;
            o[jj + 2] = (lo * sv[jj] + hi * cv[jj]) * rn;
          }
        }
        if (rr < 2) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) st16<T16>(sh.sq, warp + 8 * rr, lane + 32 * jj, o[jj]);
        } else {
          const int64_t crow =
              (((int64_t)l * p.cache_batch + p.b_off + b) * p.Hkv + g) * p.t_max + p.pos;
          T16* dstc = static_cast<T16*>(is_v ? p.v_cache : p.k_cache) + crow * kHd;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const T16 v = from_f32<T16>(o[jj]);
            dstc[lane + 32 * jj] = v;
            reinterpret_cast<T16*>(sh.kvnew)[(is_v ? kHd : 0) + lane + 32 * jj] = v;
          }
        }
      }
    }
    bar_consumers();
    trace_mark(p, k, 0);
    // ---- Q fragments (A operand) are read from shared memory per k16 step
    const uint32_t sq_base = smem_u32(sh.sq);
    const int q_row = (lane & 7) + ((lane >> 3) & 1) * 8;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    for (int j = j0; j < j1; ++j) {
      if (!ring_wait(&r.full[r.stage], r.parity, p)) return false;
      if ((j - j0) % kCons == warp) {
        uint8_t* st = r.base + (size_t)r.stage * kStage;
        const uint32_t sK = smem_u32(st), sV = sK + 4096;
        if (j == last_tile) {
          // the new row from registers; V rows past pos zeroed (their p is 0, but
          // a NaN there would still poison the product)
          for (int i = lane; i < 16 * 16; i += 32) {
            const int rr = i / 16, c16 = i % 16;
            uint4* kd = reinterpret_cast<uint4*>(st + sw_off(rr, c16));
            uint4* vd = reinterpret_cast<uint4*>(st + 4096 + sw_off(rr, c16));
            if (rr == rp) {
              *kd = reinterpret_cast<const uint4*>(sh.kvnew)[c16];
              *vd = reinterpret_cast<const uint4*>(sh.kvnew + kHd)[c16];
            } else if (rr > rp) {
              *vd = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          __syncwarp();
        }
        // S = Q K^T for 16 keys (two n8 tiles)
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int key = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t kb[4], qa[4];
            ldsm_x4(sq_base + sw_off(q_row, 2 * ks + (lane >> 4)), qa);
            ldsm_x4(sK + sw_off(key, 2 * ks + ((lane >> 3) & 1)), kb);
            mma16816<T16>(s[0], qa[0], qa[1], qa[2], qa[3], kb[0], kb[1]);
            mma16816<T16>(s[1], qa[0], qa[1], qa[2], qa[3], kb[2], kb[3]);
          }
        }
        // mask keys past pos, online softmax in the log2 domain
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = 16 * j + nt * 8 + 2 * tq + (e & 1);
            float v = s[nt][e] * p.scale_log2;
            if (key >= len) v = -INFINITY;
            s[nt][e] = v;
            mx[e >> 1] = fmaxf(mx[e >> 1], v);
          }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          const float mn = fmaxf(m_r[h], mx[h]);
          alpha[h] = ex2_approx(m_r[h] - mn);
          m_r[h] = mn;
          l_r[h] *= alpha[h];
        }
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pr[nt][e] = ex2_approx(s[nt][e] - m_r[e >> 1]);
            l_r[e >> 1] += pr[nt][e];
          }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= alpha[0];
          o[i][1] *= alpha[0];
          o[i][2] *= alpha[1];
          o[i][3] *= alpha[1];
        }
        const uint32_t pa0 = pack2<T16>(pr[0][0], pr[0][1]);
        const uint32_t pa1 = pack2<T16>(pr[0][2], pr[0][3]);
        const uint32_t pa2 = pack2<T16>(pr[1][0], pr[1][1]);
        const uint32_t pa3 = pack2<T16>(pr[1][2], pr[1][3]);
        // O += P V
        {
          const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t vb[4];
            ldsm_x4_t(sV + sw_off(key, 2 * q + (lane >> 4)), vb);
            mma16816<T16>(o[2 * q], pa0, pa1, pa2, pa3, vb[0], vb[1]);
            mma16816<T16>(o[2 * q + 1], pa0, pa1, pa2, pa3, vb[2], vb[3]);
          }
        }
        if (j == last_tile) fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[r.stage]);
      r.advance();
    }
    trace_mark(p, k, 1);
    // ---- merge the warps' states: row sums over the quad, then through smem
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
    }
    float* mw = reinterpret_cast<float*>(sh.act) + warp * (16 * kMergeStride + 32);
    float* ow = mw + 32;
    if (tq == 0) {
      mw[gq] = m_r[0];
      mw[gq + 8] = m_r[1];
      mw[16 + gq] = l_r[0];
      mw[16 + gq + 8] = l_r[1];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = i * 8 + 2 * tq;
      ow[gq * kMergeStride + c] = o[i][0];
      ow[gq * kMergeStride + c + 1] = o[i][1];
      ow[(gq + 8) * kMergeStride + c] = o[i][2];
      ow[(gq + 8) * kMergeStride + c + 1] = o[i][3];
    }
    bar_consumers();
    // partial record of this CTA for (b, g): per head [m, l, o[128]]
    int c_first, n_slots;
    attn_group(p.B * p.Hkv, T16n, bg, gridDim.x, c_first, n_slots);
    const int c_last = c_first + n_slots - 1;
    const int slot = blockIdx.x - c_first;
    float* rec = p.attn_part + ((int64_t)bg * p.attn_slots + slot) * p.rec_stride;
    float* const mall = reinterpret_cast<float*>(sh.act);
    constexpr int kWs = 16 * kMergeStride + 32;   // floats per warp's merge area
    // one thread per head: the CTA's max M and sum L, and each warp's weight
    // 2^(m_w - M), which replaces m_w in place (only this thread touches column h)
    if (tid < G) {
      const int h = tid;
      float mwv[kCons];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCons; ++w) {
        mwv[w] = mall[w * kWs + h];
        M = fmaxf(M, mwv[w]);
      }
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kCons; ++w) {
        const float sc = ex2_approx(mwv[w] - M);
        L = fmaf(sc, mall[w * kWs + 16 + h], L);
        mall[w * kWs + h] = sc;
      }
      rec[h * (kHd + 2)] = M;
      rec[h * (kHd + 2) + 1] = L;
    }
    bar_consumers();
    for (int e = tid; e < G * kHd; e += 256) {
      const int h = e / kHd, i = e % kHd;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kCons; ++w)
        v = fmaf(mall[w * kWs + h], mall[w * kWs + 32 + h * kMergeStride + i], v);
      rec[h * (kHd + 2) + 2 + i] = v;
    }
    bar_consumers();
    trace_mark(p, k, 2);
    if (tid == 0) {
      // acq_rel at GPU scope: releases this CTA's records (ordered before this
      // thread by the CTA barrier); the last arriver acquires everyone's
      unsigned int n;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(n) : "l"(p.attn_count + bg) : "memory");
      sh.flag[1] = (n == (unsigned)(c_last - c_first)) ? 1 : 0;
    }
    bar_consumers();
    if (sh.flag[1]) {
      // last CTA of (b, g): log-sum-exp merge of every slot -> att[b, heads of g].
      // The records are contiguous: read them into shared memory in one batched
      // pass, then merge from there.
      const int ns = c_last - c_first + 1;
      const float* base = p.attn_part + (int64_t)bg * p.attn_slots * p.rec_stride;
      // (a long context over few sequences can give more slots than shared memory
      // holds: then the records are read from global memory directly)
      const int scl_floats = (ns * G + 3) / 4 * 4;   // keeps the records 16-byte aligned
      const bool in_smem = ((int64_t)ns * p.rec_stride + scl_floats) * 4 <= p.act_bytes;
      float* scl = reinterpret_cast<float*>(sh.act);          // [ns][G]: exp2(m_s - M) / L
      float* recs_s = scl + scl_floats;
      auto rec_at = [&](int idx) { return in_smem ? recs_s[idx] : __ldcg(base + idx); };
      const int n4 = in_smem ? ns * p.rec_stride / 4 : 0;
      for (int i0 = tid; i0 < n4; i0 += 256 * 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * 256 < n4) v[u] = __ldcg(reinterpret_cast<const float4*>(base) + i0 + u * 256);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * 256 < n4) reinterpret_cast<float4*>(recs_s)[i0 + u * 256] = v[u];
      }
      bar_consumers();
      if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, rec_at(s2 * p.rec_stride + h * (kHd + 2)));
        float L = 0.f;
        for (int s2 = 0; s2 < ns; ++s2) {
          const int rr = s2 * p.rec_stride + h * (kHd + 2);
          const float e = ex2_approx(rec_at(rr) - M);
          scl[s2 * G + h] = e;
          L += e * rec_at(rr + 1);
        }
        const float inv = 1.f / L;
        for (int s2 = 0; s2 < ns; ++s2) scl[s2 * G + h] *= inv;
      }
      bar_consumers();
      for (int e = tid; e < G * kHd; e += 256) {
        const int h = e / kHd, i = e % kHd;
        float O = 0.f;
        for (int s2 = 0; s2 < ns; ++s2)
          O += scl[s2 * G + h] * rec_at(s2 * p.rec_stride + h * (kHd + 2) + 2 + i);
        static_cast<T16*>(p.att)[(int64_t)b * qd + (g * G + h) * kHd + i] = from_f32<T16>(O);
      }
      if (tid == 0) p.attn_count[bg] = 0u;
    }
    bar_consumers();
    trace_mark(p, k, 3);
    f += j1 - j0;
  }
  return true;
}

// ---------------------------------------------------------------- small phases
template <class TW>
__device__ void phase_embed(const Params& p) {
  const int tid = threadIdx.x - 32;
  const int64_t gt = (int64_t)blockIdx.x * 256 + tid, gs = (int64_t)gridDim.x * 256;
  for (int64_t i = gt; i < (int64_t)p.B * p.d; i += gs) {
    const int b = (int)(i / p.d), k = (int)(i % p.d);
    int id = p.tokens[b];
    if (id < 0 || id >= p.V) {
      if (k == 0) atomicOr(p.status, ST_BAD_TOKEN);
      id = 0;
    }
    p.x[(int64_t)b * p.d + k] = to_f32(static_cast<const TW*>(p.wte)[(int64_t)id * p.d + k]);
  }
}

__device__ void zero_f32(float* a, int64_t n) {
  const int tid = threadIdx.x - 32;
  const int64_t gt = (int64_t)blockIdx.x * 256 + tid, gs = (int64_t)gridDim.x * 256;
  for (int64_t i = gt * 4; i < n; i += gs * 4) {
    if (i + 4 <= n)
      *reinterpret_cast<float4*>(a + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    else
      for (int64_t k = i; k < n; ++k) a[k] = 0.f;
  }
}

template <int NT, class T16>
__device__ void phase_final_norm(const Params& p) {
  // CTA c < 8 NT: token c -> fragment entries of xnf (zeros for padding tokens)
  const int tok = blockIdx.x;
  if (tok >= 8 * NT) return;
  const int tid = threadIdx.x - 32;
  __shared__ float red[kCons];
  float s = 0.f;
  if (tok < p.B)
    for (int k = tid; k < p.d; k += 256) {
      const float v = __ldcg(p.x + (int64_t)tok * p.d + k);
      s += v * v;
    }
  s = warp_sum(s);
  if ((tid & 31) == 0) red[tid >> 5] = s;
  bar_consumers();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCons; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)p.d + p.eps);
  const int nt = tok / 8, gq = tok % 8;
  uint2* dst = reinterpret_cast<uint2*>(p.xnf);
  const int ksteps = p.d / 16;
  for (int e = tid; e < ksteps * 4; e += 256) {
    const int ks = e / 4, tq = e % 4;
    uint2 v = make_uint2(0u, 0u);
    if (tok < p.B) {
      const float* xr = p.x + (int64_t)tok * p.d + ks * 16 + 2 * tq;
      v.x = pack2<T16>(__ldcg(xr) * r, __ldcg(xr + 1) * r);
      v.y = pack2<T16>(__ldcg(xr + 8) * r, __ldcg(xr + 9) * r);
    }
    dst[((int64_t)ks * NT + nt) * 32 + gq * 4 + tq] = v;
  }
}

__device__ __forceinline__ uint64_t argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ void phase_argmax(const Params& p, const Shared& sh) {
  constexpr int kChunk = 2048;
  const int tid = threadIdx.x - 32;
  const int nch = (p.V + kChunk - 1) / kChunk;
  __shared__ unsigned long long best_w[kCons];
  for (int t = blockIdx.x; t < p.B * nch; t += gridDim.x) {
    const int b = t / nch, ch = t % nch;
    const float* row = p.logits + (int64_t)b * p.V;
    uint64_t best = 0;
    // thread: 8 consecutive logits (two 16-byte loads issued together)
    const int i0 = ch * kChunk + tid * 8;
    const int lim = min(p.V, (ch + 1) * kChunk);
    if (i0 + 8 <= lim) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(row + i0));
      const float4 c = __ldcg(reinterpret_cast<const float4*>(row + i0 + 4));
      const float v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t k = argmax_key(v[u], i0 + u);
        best = k > best ? k : best;
      }
    } else {
      for (int i = i0; i < lim; ++i) {
        const uint64_t k = argmax_key(__ldcg(row + i), i);
        best = k > best ? k : best;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if ((tid & 31) == 0) best_w[tid >> 5] = best;
    bar_consumers();
    if (tid == 0) {
      uint64_t bb = 0;
      for (int w = 0; w < kCons; ++w) bb = best_w[w] > bb ? best_w[w] : bb;
      atomicMax(p.argmax_key + b, (unsigned long long)bb);
      __threadfence();
      const unsigned int n = atomicAdd(p.argmax_count + b, 1u);
      if (n == (unsigned)(nch - 1)) {
        __threadfence();
        const uint64_t k = atomicAdd(p.argmax_key + b, 0ull);
        if (p.argmax_out) p.argmax_out[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu));
        p.argmax_count[b] = 0u;
      }
    }
    bar_consumers();
  }
}

// ================================================================== kernel
template <int NT, class T16, class TW>
__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Shared sh;
  sh.ring.base = smem;
  sh.ring.n = p.stages;
  sh.ring.stage = 0;
  sh.ring.parity = 0;
  uint8_t* q = smem + (size_t)p.stages * kStage;
  sh.act = q;
  sh.act_ksteps = p.act_bytes / (NT * 256);
  q += p.act_bytes;
  sh.xpose = reinterpret_cast<float*>(q);
  q += kXposeBytes;
  sh.sq = q;
  q += 4096;
  sh.kvnew = reinterpret_cast<uint16_t*>(q);
  q += 512;
  sh.ss_s = reinterpret_cast<float*>(q);
  q += 128;
  sh.ring.full = reinterpret_cast<uint64_t*>(q);
  sh.ring.empty = sh.ring.full + p.stages;
  sh.flag = reinterpret_cast<volatile int*>(sh.ring.empty + p.stages);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sh.ring.full[s], 1);
      mbar_init(&sh.ring.empty[s], kCons);
    }
    sh.flag[0] = sh.flag[1] = 0;
    sh.flag[2] = 1;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      producer(p, sh, &tmK, &tmV);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int nbar = 0;
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 32) p.trace[0] = global_timer_ns();
  // P0: embedding and zeroed accumulators
  phase_embed<TW>(p);
  zero_f32(p.qkv_acc, (int64_t)p.B * p.nqkv_pad);
  zero_f32(p.ss, (int64_t)2 * p.L * kMaxTok);
  zero_f32(p.logits, (int64_t)p.B * p.V);
  {
    const int tid = threadIdx.x - 32;
    const int64_t gt = (int64_t)blockIdx.x * 256 + tid;
    if (gt < kMaxTok) {
      p.argmax_key[gt] = 0ull;
      p.argmax_count[gt] = 0u;
    }
    for (int64_t i = gt; i < (int64_t)kMaxTok * p.Hkv; i += (int64_t)gridDim.x * 256)
      p.attn_count[i] = 0u;
  }
  if (!grid_barrier(p, sh, ++nbar)) return;
  for (int l = 0; l < p.L; ++l) {
    zero_f32(p.hacc, (int64_t)p.B * p.F);
    if (!consume_gemv<NT, T16>(p, sh, gemv_of(p, l, PH_QKV), nbar + 1)) return;
    if (!grid_barrier(p, sh, ++nbar)) return;
    if (l + 1 < p.L) zero_f32(p.qkv_acc + (int64_t)((l + 1) & 1) * kMaxTok * p.nqkv_pad,
                              (int64_t)p.B * p.nqkv_pad);
    if (!consume_attn<T16>(p, sh, l, nbar + 1)) return;
    if (!grid_barrier(p, sh, ++nbar)) return;
    if (!consume_gemv<NT, T16>(p, sh, gemv_of(p, l, PH_O), nbar + 1)) return;
    if (!grid_barrier(p, sh, ++nbar)) return;
    if (!consume_gemv<NT, T16>(p, sh, gemv_of(p, l, PH_FC), nbar + 1)) return;
    if (!grid_barrier(p, sh, ++nbar)) return;
    if (!consume_gemv<NT, T16>(p, sh, gemv_of(p, l, PH_PROJ), nbar + 1)) return;
    if (!grid_barrier(p, sh, ++nbar)) return;
  }
  phase_final_norm<NT, T16>(p);
  if (!grid_barrier(p, sh, ++nbar)) return;
  if (!consume_gemv<NT, T16>(p, sh, gemv_lm(p), nbar + 1)) return;
  if (!grid_barrier(p, sh, ++nbar)) return;
  phase_argmax(p, sh);
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 32)
    p.trace[2 * nbar + 1] = global_timer_ns();
}

// ===================================================================== host
// Packs rows [0, Npad) of W = [W0; W1; W2] (row-major [N, K], rows split at s0,
// s1; rows >= N zero) into 8 KB units of 128 rows x 32 columns in mma A-fragment
// order: unit (grp, kp) at ((grp * K/32 + kp) * 8192); inside it
// [kk][tile][lane] 16-byte entries holding rows grp*128 + tile*16 + {g, g + 8}
// (g = lane / 4) and columns kp*32 + kk*16 + 2(lane % 4) + {0, 1, 8, 9}.
template <class T16>
__global__ void pack_kernel(const T16* __restrict__ w0, const T16* __restrict__ w1,
                            const T16* __restrict__ w2, int s0, int s1, int N, int K, int64_t n_entries,
                            uint4* __restrict__ out) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_entries) return;
  const int lane = (int)(e & 31);
  const int tile = (int)((e >> 5) & 7);
  const int kk = (int)((e >> 8) & 1);
  const int64_t unit = e >> 9;
  const int kpairs = K / kUnitCols;
  const int grp = (int)(unit / kpairs), kp = (int)(unit % kpairs);
  const int r0 = grp * kUnitRows + tile * 16 + (lane >> 2);
  const int c0 = kp * kUnitCols + kk * 16 + 2 * (lane & 3);
  auto pair = [&](int row, int col) -> uint32_t {
    if (row >= N) return 0u;
    const T16* src = row < s0 ? w0 + (int64_t)row * K : row < s1 ? w1 + (int64_t)(row - s0) * K
                                                                  : w2 + (int64_t)(row - s1) * K;
    return *reinterpret_cast<const uint32_t*>(src + col);
  };
  out[e] = make_uint4(pair(r0, c0), pair(r0 + 8, c0), pair(r0, c0 + 8), pair(r0 + 8, c0 + 8));
}

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int64_t packed_bytes(int N, int K) { return round_up(N, kUnitRows) * K * 2; }

template <class T16>
static void pack_one(const void* w0, const void* w1, const void* w2, int s0, int s1, int N, int K,
                     uint8_t* out, cudaStream_t s) {
  const int64_t entries = packed_bytes(N, K) / 16;
  pack_kernel<T16><<<(unsigned)((entries + 255) / 256), 256, 0, s>>>(
      (const T16*)w0, (const T16*)w1, (const T16*)w2, s0, s1, N, K, entries,
      reinterpret_cast<uint4*>(out));
}

nc_status pack_weights(const PackSrc& src, bool half, uint8_t* out, cudaStream_t s) {
  const int d = src.d, qd = src.H * kHd, kvd = src.Hkv * kHd, F = src.F;
  const int nqkv = qd + 2 * kvd;
  const int64_t b_qkv = packed_bytes(nqkv, d), b_o = packed_bytes(d, qd), b_fc = packed_bytes(F, d),
                b_proj = packed_bytes(d, F);
  const int64_t layer = b_qkv + b_o + b_fc + b_proj;
  for (int l = 0; l < src.L; ++l) {
    uint8_t* lw = out + l * layer;
    if (half) {
      pack_one<f16>(src.wq[l], src.wk[l], src.wv[l], qd, qd + kvd, nqkv, d, lw, s);
      pack_one<f16>(src.wo[l], src.wo[l], src.wo[l], INT32_MAX, INT32_MAX, d, qd, lw + b_qkv, s);
      pack_one<f16>(src.wfc[l], src.wfc[l], src.wfc[l], INT32_MAX, INT32_MAX, F, d, lw + b_qkv + b_o, s);
      pack_one<f16>(src.wproj[l], src.wproj[l], src.wproj[l], INT32_MAX, INT32_MAX, d, F,
                    lw + b_qkv + b_o + b_fc, s);
    } else {
      pack_one<bf16>(src.wq[l], src.wk[l], src.wv[l], qd, qd + kvd, nqkv, d, lw, s);
      pack_one<bf16>(src.wo[l], src.wo[l], src.wo[l], INT32_MAX, INT32_MAX, d, qd, lw + b_qkv, s);
      pack_one<bf16>(src.wfc[l], src.wfc[l], src.wfc[l], INT32_MAX, INT32_MAX, F, d, lw + b_qkv + b_o, s);
      pack_one<bf16>(src.wproj[l], src.wproj[l], src.wproj[l], INT32_MAX, INT32_MAX, d, F,
                     lw + b_qkv + b_o + b_fc, s);
    }
  }
  uint8_t* lm = out + src.L * layer;
  if (half)
    pack_one<f16>(src.lm, src.lm, src.lm, INT32_MAX, INT32_MAX, src.V, d, lm, s);
  else
    pack_one<bf16>(src.lm, src.lm, src.lm, INT32_MAX, INT32_MAX, src.V, d, lm, s);
  count_launches(4 * src.L + 1);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

Layout layout_of(int L, int d, int H, int Hkv, int F, int V) {
  Layout lo{};
  const int qd = H * kHd, kvd = Hkv * kHd;
  lo.nqkv = qd + 2 * kvd;
  lo.nqkv_pad = (int)round_up(lo.nqkv, kUnitRows);
  lo.vpad = (int)round_up(V, kUnitRows);
  lo.off_o = packed_bytes(lo.nqkv, d);
  lo.off_fc = lo.off_o + packed_bytes(d, qd);
  lo.off_proj = lo.off_fc + packed_bytes(F, d);
  lo.layer_bytes = lo.off_proj + packed_bytes(d, F);
  lo.total_bytes = lo.layer_bytes * L + packed_bytes(V, d);
  return lo;
}

bool supported(int d, int H, int Hkv, int F, int hd) {
  return hd == kHd && H % Hkv == 0 && H / Hkv <= 16 && d % kUnitRows == 0 && F % kUnitRows == 0 &&
         (H * kHd) % kUnitCols == 0;
}

// Largest number of partial-state slots any (sequence, KV head) gets.
int attn_slots_needed(int B, int Hkv, int pos, int P) {
  const int T16 = (pos + 1 + 15) / 16;
  int best = 1;
  for (int bg = 0; bg < B * Hkv; ++bg) {
    int c_first, ns;
    attn_group(B * Hkv, T16, bg, P, c_first, ns);
    best = std::max(best, ns);
  }
  return best;
}

size_t smem_bytes(int nt, int d, int* stages, int* act_bytes) {
  const int ksteps = d / 16;
  int act = std::max(nt * 256 * ksteps, kMergeBytes);
  act = (act + 1023) / 1024 * 1024;
  const int fixed = 1024 /*align*/ + kXposeBytes + 4096 + 512 + 128 + 64;
  const int limit = 232448 - 1024;   // dynamic part; static shared memory is small
  int st = (limit - fixed - act) / (kStage + 16);
  if (st > 24) st = 24;
  *stages = st;
  *act_bytes = act;
  return (size_t)st * kStage + act + fixed + 16 * st;
}

template <int NT, class T16, class TW>
static nc_status launch_t(const CUtensorMap& tk, const CUtensorMap& tv, Params p, int sms,
                          size_t smem, cudaStream_t s) {
  auto kern = decode_step_kernel<NT, T16, TW>;
  if (!ensure_dyn_smem((const void*)kern, smem)) return NC_ERR_CUDA;
  void* args[] = {(void*)&tk, (void*)&tv, (void*)&p};
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(sms), dim3(kThreads),
                                                    args, smem, s);
  count_launches(1);
  if (e != cudaSuccess) {
    set_last_error("decode step launch failed: %s", cudaGetErrorString(e));
    return NC_ERR_CUDA;
  }
  return NC_OK;
}

template <int NT>
static nc_status launch_nt(const CUtensorMap& tk, const CUtensorMap& tv, const Params& p, bool half,
                           nc_dtype wdt, int sms, size_t smem, cudaStream_t s) {
  if (half) {
    if (wdt == NC_BF16) return launch_t<NT, f16, bf16>(tk, tv, p, sms, smem, s);
    if (wdt == NC_F16) return launch_t<NT, f16, f16>(tk, tv, p, sms, smem, s);
    return launch_t<NT, f16, float>(tk, tv, p, sms, smem, s);
  }
  if (wdt == NC_BF16) return launch_t<NT, bf16, bf16>(tk, tv, p, sms, smem, s);
  if (wdt == NC_F16) return launch_t<NT, bf16, f16>(tk, tv, p, sms, smem, s);
  return launch_t<NT, bf16, float>(tk, tv, p, sms, smem, s);
}

nc_status launch_step(const CUtensorMap& tk, const CUtensorMap& tv, Params p, bool half,
                      nc_dtype wdt, int sms, cudaStream_t s) {
  const int nt = p.B <= 8 ? 1 : (p.B <= 16 ? 2 : 4);
  int stages = 0, act = 0;
  const size_t smem = smem_bytes(nt, p.d, &stages, &act);
  if (stages < 4) {
    set_last_error("decode step: shared memory too small for the ring (%d stages)", stages);
    return NC_ERR_UNSUPPORTED;
  }
  p.stages = stages;
  p.act_bytes = act;
  if (nt == 1) return launch_nt<1>(tk, tv, p, half, wdt, sms, smem, s);
  if (nt == 2) return launch_nt<2>(tk, tv, p, half, wdt, sms, smem, s);
  return launch_nt<4>(tk, tv, p, half, wdt, sms, smem, s);
}

}  // namespace dec
}  // namespace nc

namespace nc {
namespace dec {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D view [rows, 128] of a 16-bit KV array, boxes of 16 rows x 64 columns with
// the 128-byte swizzle (the layout the attention phase reads).
bool make_cache_map(CUtensorMap* map, void* base, uint64_t rows, bool half) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dec
}  // namespace nc
