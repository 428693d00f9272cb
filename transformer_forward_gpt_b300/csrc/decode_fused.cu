// One decode step of the whole model in one persistent launch (16-bit path,
// head_dim 128, up to 32 sequences per launch).
//
// Decode is bound by HBM: every step streams all projection weights and every
// cached K/V row once, and each of them is used by only B <= 32 tokens. With one
// kernel per projection the step pays a launch, a ramp and a tail per kernel
// (about 180 of them for a 20-layer model), which costs more than the streaming
// itself. Here one CTA per SM runs the whole step with four roles:
//
//   warp 0 (producer)   one thread streams the CTA's share of every weight
//                       matrix (pre-swizzled 16 KB units, 1-D bulk copies) and of
//                       the KV cache (2-D TMA tiles of 32 positions, 128-byte
//                       swizzle) into a ring of 16 KB stages. Nothing it loads
//                       depends on the step's activations, so it runs ahead
//                       across the grid barriers of the phases.
//   warps 1 and 10      the MMA issuers (one thread each; warp 1 allocates the
//                       TMEM): tcgen05.mma for every weight unit of the
//                       projection phases, the unit's 128 weight rows the A
//                       operand (M = 128), the 32 token rows staged by the
//                       consumers the B operand (N = 32), fp32 accumulation in
//                       TMEM over the CTA's K range. Issuer i takes the units at
//                       ring positions of parity i (see mma_gemv).
//   warps 2..9          consumers, phase by phase, separated by grid barriers:
//     P0       embedding x = wte[token]; zero the accumulators of the step
//     per layer:
//       QKV    acc = x Wqkv^T (x un-normalised: RMSNorm has no gain, so the
//              norm is one scale per token, applied after the barrier); the CTAs
//              that cover feature group 0 also sum x^2 for that scale
//       ATTN   RoPE + QK norm of q and of the new k, cache write of the new
//              k / v, split-KV attention over positions 0..pos (all query heads
//              of a KV head share one pass over K/V); each CTA adds its
//              softmax sums, weighted against a fixed reference, into
//              accumulators that the CTAs of a (sequence, KV head) share
//       O      x += att Wo^T, att = numerators / denominators while staging
//       FC     hacc = x Wfc^T (un-normalised, sum of x^2 as in QKV)
//       PROJ   x += relu(r hacc)^2 Wproj^T
//     FNORM    xn = RMSNorm(x), written as the B operand image of the LM head
//     LM       logits = xn Wlm^T
//     ARGMAX   greedy token per sequence (lowest index on ties)
//
// Projection phases: the weight matrix [N, K] is cut into units of 128 rows x 64
// columns (16 KB, stored in the 128-byte-swizzled K-major layout the tensor core
// reads). Units are ordered row-group-major and each CTA takes an equal
// contiguous range of them, so every CTA streams the same number of bytes. The
// consumers first stage the 64-column chunks of the activations the range needs
// (32 token rows, 16-bit, same swizzle); the MMA issuers then run the range,
// one accumulator per issuer and row group it touches; the consumers read each finished
// accumulator from TMEM and add it into the fp32 output with reductions.
// Projection outputs therefore sum in a run-dependent order (fp32).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "nc_internal.h"
#include "decode_fused.h"

namespace nc {
namespace dec {

constexpr int kCons = 8;                    // consumer warps (CTA warps 2..9)
constexpr int kThreads = 32 * (3 + kCons);  // producer, MMA issuer 0, consumers, MMA issuer 1
constexpr int kStage = 16384;               // bytes of one ring stage
constexpr int kUnitRows = 128;              // weight rows of one unit (MMA M)
constexpr int kUnitCols = 64;               // weight columns of one unit (128 bytes)
constexpr int kTok = kMaxTok;               // token rows of a B chunk (MMA N)
constexpr int kChunkBytes = kTok * 128;     // one 64-column chunk of kTok tokens
constexpr int kHd = 128;
constexpr int kKeys = 32;                   // positions per K/V tile
constexpr int kMergeStride = 132;           // floats per row of a warp's merge area
// Partial softmax states are combined with weights 2^(m - kScoreRef). QK
// RMS-norm makes |q.k| <= head_dim, so a score (log2 units, scale 1/sqrt(hd)
// folded in) is at most sqrt(128) * log2(e) = 16.3 in magnitude: every weight
// lies in [2^-37, 2^-3.6], far inside fp32, and no maximum has to be found first.
constexpr float kScoreRef = 20.f;
constexpr int kMergeBytes = kCons * (16 * kMergeStride + 32) * 4;
// Tensor memory: per MMA issuer two alternating accumulators (issuer i, run
// parity a at column (a + 2 i) kTok); in sampling mode the LM head's row groups
// that the CTA keeps until the draw take one accumulator each from column
// kTmemResident on (issuer 1 is idle then, so they may cover its columns).
constexpr int kTmemResident = 2 * kTok;
constexpr int kTmemCols = 256;
static_assert(kTmemResident + kMaxResidentGroups * kTok <= kTmemCols, "TMEM columns");

enum Phase : int { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_FC = 3, PH_PROJ = 4 };
// Activation sources of a projection: fp32 x (+ sum of squares), fp32 FC sums
// (scaled, ReLU^2), the attention phase's summed numerators and denominators
// (divided while staged), or an image already in the B-chunk layout (final norm).
enum ActKind : int { ACT_X32 = 0, ACT_H32 = 1, ACT_ATT = 2, ACT_IMG = 3 };

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

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
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

// Byte offset of 16-byte chunk c16 (8 values) of row r in a [R rows x 128 values]
// tile stored as two 64-column halves of R x 128 bytes with the 128-byte swizzle
// (chunk index XOR row % 8 inside each 1 KB group of 8 rows): the layout a TMA
// box of 64 columns x R rows lands in. R = 16 for the Q tile, 32 for K/V tiles.
template <int R>
__device__ __forceinline__ uint32_t sw_off(int r, int c16) {
  return (uint32_t)((c16 >> 3) * (R * 128) + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}
// Byte offset of 16-byte chunk j of token row t inside one B chunk (kTok rows x
// 128 bytes, 128-byte swizzle): the layout of the MMA's K-major B operand.
__host__ __device__ __forceinline__ uint32_t bchunk_off(int t, int j) {
  return (uint32_t)((t >> 3) * 1024 + (t & 7) * 128 + ((j ^ (t & 7)) << 4));
}

// ------------------------------------------------------------ work ranges
// Contiguous share [lo, hi) of `total` items for CTA c of P. With fewer items
// than CTAs, CTA c < total takes item c; otherwise every share is non-empty. So
// the CTAs that touch any run of consecutive items are consecutive themselves.
// 32-bit arithmetic throughout (the host checks total * P < 2^31): 64-bit
// division is a long software routine, and this code runs on every phase.
__host__ __device__ __forceinline__ void share(int total, int c, int P, int& lo, int& hi) {
  if (total < P) {
    lo = c < total ? c : total;
    hi = c + 1 < total ? c + 1 : total;
  } else {
    lo = (int)((unsigned)(total * c) / (unsigned)P);
    hi = (int)((unsigned)(total * (c + 1)) / (unsigned)P);
  }
}

// Attention work: tiles of kKeys positions over (sequence, KV head) pairs bg =
// b * Hkv + g; sequence b attends over positions 0..pos[b], so each of its pairs
// has tiles_of(b) tiles. Tiles are numbered pair after pair (f). With per-pair
// CTA blocks every CTA holds one contiguous tile range of one pair (one partial
// state per CTA); otherwise CTA c holds an even share of all tiles.
// attn_work gives CTA c's range [f0, f1).
__host__ __device__ __forceinline__ int tiles_of(const Params& p, int b) {
  return (p.pos[b] + kKeys) / kKeys;
}
__host__ __device__ __forceinline__ int tile0_of(const Params& p, int bg) {
  const int b = (int)((unsigned)bg / (unsigned)p.Hkv);
  return p.tile_pre[b] + (bg - b * p.Hkv) * tiles_of(p, b);
}
// pair of tile f, and f's index j within the pair
__device__ __forceinline__ int pair_at(const Params& p, int f, int& j) {
  int lo = 0, hi = p.B;   // tile_pre[lo] <= f < tile_pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_pre[mid] <= f) lo = mid; else hi = mid;
  }
  f -= p.tile_pre[lo];
  const int nt = tiles_of(p, lo);
  const int g = (int)((unsigned)f / (unsigned)nt);
  j = f - g * nt;
  return lo * p.Hkv + g;
}
__host__ __device__ __forceinline__ void attn_work(const Params& p, int c, int P, int& f0, int& f1) {
  if (p.attn_blocks) {
    // the pair whose block holds c: pair_c0 increases strictly from 0 to P
    int lo = 0, hi = p.B * p.Hkv;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.pair_c0[mid] <= c) lo = mid; else hi = mid;
    }
    const int cs = p.pair_c0[lo], ce = p.pair_c0[lo + 1];
    const int nt = tiles_of(p, (int)((unsigned)lo / (unsigned)p.Hkv));
    int j0, j1;
    share(nt, c - cs, ce - cs, j0, j1);
    const int t0 = tile0_of(p, lo);
    f0 = t0 + j0;
    f1 = t0 + j1;
  } else {
    share(p.attn_total, c, P, f0, f1);
  }
}

// ------------------------------------------------------------------- state
// A position in the ring of stages; every role keeps its own copy.
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
  __device__ __forceinline__ void skip(int k) {
    const unsigned s = (unsigned)(stage + k), q = s / (unsigned)n;
    stage = (int)(s - q * (unsigned)n);
    parity ^= q & 1u;
  }
  // stage and parity of the position k ahead of this one
  __device__ __forceinline__ void ahead(int k, int& st, uint32_t& par) const {
    const unsigned s = (unsigned)(stage + k), q = s / (unsigned)n;
    st = (int)(s - q * (unsigned)n);
    par = parity ^ (q & 1u);
  }
};

struct Shared {
  Ring ring;
  uint8_t* act;          // B chunks of the projection phases / attention merge area
  uint8_t* sq;           // Q tiles of up to two pairs (16 x 128 each, swizzled)
  uint16_t* kvnew;       // new K row, new V row of up to two pairs (16-bit)
  uint64_t* acc_full;    // [2] accumulator ready (tcgen05.commit)
  uint64_t* acc_empty;   // [2] accumulator read by the consumers (8 arrivals)
  uint64_t* b_full;      // B chunks staged (8 arrivals)
  uint64_t* fin;         // the MMA issuers' last commits (2 arrivals)
  uint32_t* tmem_slot;
  volatile int* flag;    // [2] barrier ok
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
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 64)
    p.trace[2 * p.nbar + 2 + 6 * (k - 1) + m] = global_timer_ns();
}
// Producer mark: when CTA 0's producer starts issuing the loads of the phase
// that ends at grid barrier k.
__device__ __forceinline__ void trace_producer(const Params& p, int k) {
  if (p.trace && blockIdx.x == 0) p.trace[2 * p.nbar + 2 + 6 * (k - 1) + 4] = global_timer_ns();
}

// A wait reads the abort word (an L2 round trip) only once it has lasted this
// long, so the common, short waits poll nothing but their own condition.
constexpr uint64_t kAbortCheckNs = 20000;

// Bounded wait on an mbarrier phase; false on timeout (which raises the abort
// word) or when another CTA or role has aborted the step.
__device__ bool bwait_slow(uint64_t* bar, uint32_t parity, const Params& p) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    const uint64_t dt = global_timer_ns() - t0;
    if (dt > kAbortCheckNs && aborted(p)) return false;
    if (dt > kWaitLimitNs) {
      raise_abort(p);
      return false;
    }
  }
}
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, const Params& p) {
  return mbar_try_wait(bar, parity) || bwait_slow(bar, parity, p);
}

// Grid barrier number k (1-based) of this launch among the consumer warps of all
// CTAs. Returns false (in every consumer thread of the CTA) if the step was
// aborted.
__device__ bool grid_barrier(const Params& p, const Shared& sh, int k) {
  bar_consumers();
  const int tid = threadIdx.x - 64;
  if (tid == 0) {
    // an aborted step is noticed in the wait below (its slow path): a read of the
    // abort word here would hold up the release by a round trip to L2
    bool ok = true;
    const bool tr = p.trace && blockIdx.x == 0;
    uint64_t t_arr = 0;
    if (p.trace) t_arr = global_timer_ns();
    if (tr) p.trace[2 * k - 1] = t_arr;
    // release at GPU scope: this CTA's writes (ordered before this thread by the
    // CTA barrier above) are visible to any CTA that acquires the count
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p.bar_counter) : "memory");
    const unsigned long long target = p.bar_base + (unsigned long long)k * gridDim.x;
    const uint64_t t0 = global_timer_ns();
    int it = 0;
    while (ok && ld_acquire_u64(p.bar_counter) < target) {
      if (++it == 16) {
        it = 0;
        const uint64_t dt = global_timer_ns() - t0;
        if (dt > kAbortCheckNs && aborted(p)) {
          ok = false;
          break;
        }
        if (dt > kWaitLimitNs) {
          raise_abort(p);
          ok = false;
          break;
        }
      }
    }
    sh.flag[2] = ok ? 1 : 0;
    if (p.trace) {
      const uint64_t t_exit = global_timer_ns();
      if (tr) p.trace[2 * k] = t_exit;
      if (blockIdx.x < kTraceCtas) {
        unsigned long long* c = p.trace + 8 * p.nbar + 2 + ((k - 1) * kTraceCtas + blockIdx.x) * 2;
        c[0] = t_arr;
        c[1] = t_exit;
      }
    }
  }
  bar_consumers();
  return sh.flag[2] != 0;
}

// --------------------------------------------------------- phase geometry
struct Gemv {
  const uint8_t* w;    // packed units
  int groups, nch;     // units = groups * nch (nch 64-column chunks per row group)
  float* out;          // fp32 [B, ldo]
  int ldo, n_valid;
  int act_kind;
  const void* act;     // source of the activations
  int act_ld;          // row pitch (elements) of an fp32 source
  const float* ss_in;  // ACT_H32: sums of squares giving the per-token scale
  float* ss_out;       // ACT_X32: sums of squares of x accumulated here (or null)
  const float* den;    // ACT_ATT: softmax denominators [kMaxTok][H]
  int whole;           // 1: CTAs take whole row groups (LM head, sampling mode)
};

__device__ __forceinline__ Gemv gemv_of(const Params& p, int l, int ph) {
  Gemv g{};
  const uint8_t* lw = p.wpack + (int64_t)l * p.layer_bytes;
  const int d = p.d, qd = p.H * kHd;
  switch (ph) {
    case PH_QKV:
      g.w = lw;
      g.groups = p.nqkv_pad / kUnitRows;
      g.nch = d / kUnitCols;
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
      g.nch = qd / kUnitCols;
      g.out = p.x;
      g.ldo = d;
      g.n_valid = d;
      g.act_kind = ACT_ATT;
      g.act = p.att_num + (int64_t)(l & 1) * kMaxTok * qd;
      g.act_ld = qd;
      g.den = p.att_den + (l & 1) * kMaxTok * p.H;
      break;
    case PH_FC:
      g.w = lw + p.off_fc;
      g.groups = p.F / kUnitRows;
      g.nch = d / kUnitCols;
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
      g.nch = p.F / kUnitCols;
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
  g.nch = p.d / kUnitCols;
  g.out = p.logits;
  g.ldo = p.V;
  g.n_valid = p.V;
  g.act_kind = ACT_IMG;
  g.act = p.xn_img;
  g.whole = p.sample;
  return g;
}

// The step as one sequence of phases q = 5 l + ph (ph a Phase of layer l), then
// q = 5 L (final norm) and q = 5 L + 1 (LM head). Every role walks it in one
// loop with one call site per kind of phase: the kernel's code stays small
// enough that the phases share their instructions in the instruction cache.
__device__ __forceinline__ int phase_layer(int q, int& ph) {
  const int l = (int)((unsigned)q / 5u);
  ph = q - 5 * l;
  return l;
}

// The CTA's unit range of a projection and the B chunk slot of each unit: a
// range shorter than a row group holds distinct chunks, staged in range order;
// a longer one needs every chunk, staged in chunk order.
struct Range {
  int u0, u1;
  int nslots;
  bool all;
  int c0;   // chunk of unit u0 (u0 % nch)
  int g0;   // row group of unit u0
  __device__ __forceinline__ int chunk(int s, int nch) const {
    if (all) return s;
    const int c = c0 + s;
    return c < nch ? c : c - nch;   // a short range wraps at most once
  }
};
__device__ __forceinline__ Range range_of(const Gemv& g) {
  Range r;
  if (g.whole) {
    int g0, g1;
    share(g.groups, blockIdx.x, gridDim.x, g0, g1);
    r.u0 = g0 * g.nch;
    r.u1 = g1 * g.nch;
  } else {
    share(g.groups * g.nch, blockIdx.x, gridDim.x, r.u0, r.u1);
  }
  r.all = r.u1 - r.u0 >= g.nch;
  r.nslots = r.all ? g.nch : r.u1 - r.u0;
  r.g0 = (int)((unsigned)r.u0 / (unsigned)g.nch);
  r.c0 = r.u0 - r.g0 * g.nch;
  return r;
}

// ================================================================ producer
__device__ void produce_gemv(const Params& p, Ring& r, const Gemv& g, uint64_t pol, bool& ok) {
  const Range rg = range_of(g);
  for (int u = rg.u0; u < rg.u1 && ok; ++u) {
    if (!bwait(&r.empty[r.stage], r.parity ^ 1u, p)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&r.full[r.stage], kStage);
    bulk_load(r.base + (size_t)r.stage * kStage, g.w + (size_t)u * kStage, kStage, &r.full[r.stage], pol);
    r.advance();
  }
}

__device__ void produce_attn(const Params& p, Ring& r, const CUtensorMap* tk, const CUtensorMap* tv,
                             int l, uint64_t pol, bool& ok) {
  int f0, f1;
  attn_work(p, blockIdx.x, gridDim.x, f0, f1);
  int j = 0;
  int bg = f0 < f1 ? pair_at(p, f0, j) : 0;
  int nt = tiles_of(p, (int)((unsigned)bg / (unsigned)p.Hkv));
  for (int f = f0; f < f1 && ok; ++f, ++j) {
    if (j == nt) {
      j = 0;
      ++bg;
      nt = tiles_of(p, (int)((unsigned)bg / (unsigned)p.Hkv));
    }
    const int b = (int)((unsigned)bg / (unsigned)p.Hkv), g = bg - b * p.Hkv;
    const int64_t row =
        (((int64_t)l * p.cache_batch + p.b_off + b) * p.Hkv + g) * p.t_max + kKeys * j;
    if (!bwait(&r.empty[r.stage], r.parity ^ 1u, p)) {
      ok = false;
      break;
    }
    uint8_t* dst = r.base + (size_t)r.stage * kStage;
    mbar_arrive_expect_tx(&r.full[r.stage], kStage);
    tma_load_2d_hint(dst, tk, &r.full[r.stage], 0, (int32_t)row, pol);
    tma_load_2d_hint(dst + 4096, tk, &r.full[r.stage], 64, (int32_t)row, pol);
    tma_load_2d_hint(dst + 8192, tv, &r.full[r.stage], 0, (int32_t)row, pol);
    tma_load_2d_hint(dst + 12288, tv, &r.full[r.stage], 64, (int32_t)row, pol);
    r.advance();
  }
}

__device__ void producer(const Params& p, Ring r, const CUtensorMap* tk, const CUtensorMap* tv) {
  const uint64_t pol = l2_policy_evict_first();
  bool ok = true;
  // phase q ends at grid barrier q + 2 (barrier 1 ends the embedding); the final
  // norm streams nothing
#pragma unroll 1
  for (int q = 0; q < 5 * p.L + 2 && ok; ++q) {
    int ph;
    const int l = phase_layer(q, ph);
    if (l == p.L && ph == 0) continue;
    trace_producer(p, q + 2);
    if (l < p.L && ph == PH_ATTN)
      produce_attn(p, r, tk, tv, l, pol, ok);
    else
      produce_gemv(p, r, l < p.L ? gemv_of(p, l, ph) : gemv_lm(p), pol, ok);
  }
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

// ==================================================================== MMA
// Issues the MMAs of one projection phase: per row group of the CTA's range one
// run of units, per unit four K = 16 steps. Two issuer threads share a phase
// (one tcgen05.mma takes about as long to issue as to run at N = 32, so two
// issuers nearly double the rate): with an even number of ring stages, issuer i
// takes the units at ring positions of parity i, so every stage has one issuer,
// and sums them in its own accumulator of the run. In whole-group mode (sampling)
// issuer 0 takes every unit into the run's resident accumulator. Both commit
// every run's accumulator barrier (an issuer without units of the run commits
// at once).
template <class T16>
__device__ bool mma_gemv(const Params& p, const Shared& sh, Ring& r, const Gemv& g,
                         uint32_t tmem_base, int& run, uint32_t& bphase, int issuer) {
  const Range rg = range_of(g);
  if (rg.u0 >= rg.u1) return true;
  if (!bwait(sh.b_full, bphase & 1u, p)) return false;
  ++bphase;
  tc_fence_after();
  constexpr uint32_t kIdesc = idesc_f32acc(Fmt16<T16>::code, kUnitRows, kTok);
  const uint32_t act = smem_u32(sh.act);
  // runs: one per row group of the range; slots in range order (or by chunk)
  int u = rg.u0, kp = rg.c0, sl = 0, rr = 0;
  while (u < rg.u1) {
    const int n = min(g.nch - kp, rg.u1 - u);
    const int a = run & 1;
    if (!bwait(&sh.acc_empty[a], ((run >> 1) & 1) ^ 1u, p)) return false;
    tc_fence_after();
    const uint32_t d = g.whole ? tmem_base + kTmemResident + (rr++) * kTok
                               : tmem_base + (uint32_t)(a + 2 * issuer) * kTok;
    int mine = 0;
    for (int i = 0; i < n; ++i, ++sl) {
      const bool own = g.whole ? issuer == 0 : (r.stage & 1) == issuer;
      if (own) {
        if (!bwait(&r.full[r.stage], r.parity, p)) return false;
        tc_fence_after();
        const uint64_t wd = sdesc_kmajor_sw128(smem_u32(r.base + (size_t)r.stage * kStage));
        const uint64_t bd = sdesc_kmajor_sw128(act + (rg.all ? kp + i : sl) * kChunkBytes);
        // +32 bytes along K per step: +2 in the descriptor's address field
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16kind_ss(d, wd + 2 * k, bd + 2 * k, kIdesc, (mine > 0 || k > 0) ? 1u : 0u);
        mma_commit(&r.empty[r.stage]);
        ++mine;
      }
      r.advance();
    }
    mma_commit(&sh.acc_full[a]);
    ++run;
    u += n;
    kp = 0;
  }
  return true;
}

template <class T16>
__device__ void mma_role(const Params& p, const Shared& sh, Ring r, uint32_t tmem_base, int issuer) {
  int run = 0;
  uint32_t bphase = 0;
  bool ok = true;
  int f0, f1;   // the attention phase's stages belong to the consumers
  attn_work(p, blockIdx.x, gridDim.x, f0, f1);
#pragma unroll 1
  for (int q = 0; q < 5 * p.L + 2 && ok; ++q) {
    int ph;
    const int l = phase_layer(q, ph);
    if (l == p.L && ph == 0) continue;
    if (l < p.L && ph == PH_ATTN)
      r.skip(f1 - f0);
    else
      ok = mma_gemv<T16>(p, sh, r, l < p.L ? gemv_of(p, l, ph) : gemv_lm(p), tmem_base, run, bphase,
                         issuer);
  }
  // every MMA of both issuers has completed once both commits have arrived
  mma_commit(sh.fin);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(sh.fin, 0)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// =============================================================== consumers
// Stages the B chunks of the CTA's range: token rows 0..kTok-1 (zeros past B),
// 64 columns each, 16-bit, in the MMA's swizzled K-major layout. For ACT_X32
// the squares of the columns of row group 0 in the range are summed and added
// to g.ss_out; for ACT_H32 each value becomes relu(r * h)^2 with the token's
// norm scale r. Ends with the B-full arrival of each consumer warp.
template <class T16>
__device__ void stage_b(const Params& p, const Shared& sh, const Gemv& g, const Range& rg) {
  const int tid = threadIdx.x - 64;
  const int lane = tid & 31;
  if (g.act_kind == ACT_IMG) {
    // the image already has the chunk layout: 16-byte copies, eight in flight
    constexpr int kPer = kChunkBytes / 16;
    const uint4* src = static_cast<const uint4*>(g.act);
    uint4* dst = reinterpret_cast<uint4*>(sh.act);
    const int total = rg.nslots * kPer;
    for (int i0 = tid; i0 < total; i0 += 256 * 8) {
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * 256;
        v[q] = make_uint4(0u, 0u, 0u, 0u);
        if (i < total) v[q] = __ldcg(src + (int64_t)rg.chunk(i / kPer, g.nch) * kPer + i % kPer);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * 256;
        if (i < total) dst[i] = v[q];
      }
    }
  } else if (g.act_kind == ACT_ATT) {
    // token tok, 16-byte chunk j of every slot: eight values of head c / 2's
    // attention output (values 64 (c % 2) + 8 j ..), the summed numerators over
    // the head's summed denominator; the loads of up to eight slots in flight
    const int tok = tid >> 3, j = tid & 7;
    const bool tok_ok = tok < p.B;
    const float* src = static_cast<const float*>(g.act) + (int64_t)tok * g.act_ld + 8 * j;
    const float* den = g.den + tok * p.H;
    uint8_t* dst = sh.act + bchunk_off(tok, j);
    for (int s0 = 0; s0 < rg.nslots; s0 += 8) {
      float4 a[8], b[8];
      float dn[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int s = s0 + q;
        a[q] = b[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        dn[q] = 1.f;
        if (s < rg.nslots && tok_ok) {
          const int c = rg.chunk(s, g.nch);
          const float* sp = src + c * kUnitCols;
          a[q] = __ldcg(reinterpret_cast<const float4*>(sp));
          b[q] = __ldcg(reinterpret_cast<const float4*>(sp + 4));
          dn[q] = __ldcg(den + (c >> 1));
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int s = s0 + q;
        if (s >= rg.nslots) continue;
        const float inv = 1.f / dn[q];
        *reinterpret_cast<uint4*>(dst + (size_t)s * kChunkBytes) =
            make_uint4(pack2<T16>(a[q].x * inv, a[q].y * inv), pack2<T16>(a[q].z * inv, a[q].w * inv),
                       pack2<T16>(b[q].x * inv, b[q].y * inv), pack2<T16>(b[q].z * inv, b[q].w * inv));
      }
    }
  } else {
    // thread: token tok = tid / 8, 16-byte chunk j = tid % 8 of every slot; the
    // loads of up to eight slots are in flight at once
    const int tok = tid >> 3, j = tid & 7;
    const bool tok_ok = tok < p.B;
    const float* src = static_cast<const float*>(g.act) + (int64_t)tok * g.act_ld + 8 * j;
    const bool want_ss = g.act_kind == ACT_X32 && g.ss_out != nullptr;
    float rscale = 0.f;
    if (g.act_kind == ACT_H32 && tok_ok) rscale = rsqrtf(__ldcg(g.ss_in + tok) / (float)p.d + p.eps);
    float ssum = 0.f, amax = 0.f;
    uint8_t* dst = sh.act + bchunk_off(tok, j);
    for (int s0 = 0; s0 < rg.nslots; s0 += 8) {
      float4 a[8], b[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int s = s0 + q;
        a[q] = b[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < rg.nslots && tok_ok) {
          const float* sp = src + rg.chunk(s, g.nch) * kUnitCols;
          a[q] = __ldcg(reinterpret_cast<const float4*>(sp));
          b[q] = __ldcg(reinterpret_cast<const float4*>(sp + 4));
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int s = s0 + q;
        if (s >= rg.nslots) continue;
        float v[8] = {a[q].x, a[q].y, a[q].z, a[q].w, b[q].x, b[q].y, b[q].z, b[q].w};
        if (want_ss) {
          // row group 0's units of the range: the first ones (u0 + s < nch), or,
          // for a range holding every chunk, chunks from u0 on
          const bool rg0 = rg.all ? (rg.u0 < g.nch && s >= rg.u0) : (rg.u0 + s < g.nch);
          if (rg0)
#pragma unroll
            for (int e = 0; e < 8; ++e) ssum = fmaf(v[e], v[e], ssum);
        }
        if (g.act_kind == ACT_H32) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float t = fmaxf(v[e] * rscale, 0.f);
            v[e] = t * t;
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        *reinterpret_cast<uint4*>(dst + (size_t)s * kChunkBytes) =
            make_uint4(pack2<T16>(v[0], v[1]), pack2<T16>(v[2], v[3]), pack2<T16>(v[4], v[5]),
                       pack2<T16>(v[6], v[7]));
      }
    }
    note_range<T16>(amax, p.status);   // x is staged un-normalised
    if (want_ss) {
      // the eight lanes of a token are adjacent
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 4);
      if (j == 0 && tok_ok && ssum != 0.f) red_add_f32(g.ss_out + tok, ssum);   // no return value
    }
  }
  // generic-proxy stores become visible to the tensor core (async proxy)
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(sh.b_full);
}

// Consumer side of a projection phase: stage the B chunks, then read every
// accumulator the MMA issuers finish and add it into the output. Warp w of the
// consumers reads TMEM lane quarter (w + 2) % 4 (the quarter its CTA warp index
// may access) and token columns 16 * (w / 4) .. + 15.
template <class T16>
__device__ bool consume_gemv(const Params& p, Shared& sh, const Gemv& g, int k, uint32_t tmem_base,
                             int& run) {
  const Range rg = range_of(g);
  if (rg.u0 >= rg.u1) return true;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4, half = (warp - 2) / 4;
  trace_mark(p, k, 3);
  stage_b<T16>(p, sh, g, rg);
  trace_mark(p, k, 0);
  bool ok = true;
  int u = rg.u0, grp = rg.g0, kp = rg.c0;
  int par = sh.ring.stage & 1;   // ring position parity of the unit u (even ring)
  while (u < rg.u1) {
    const int n = min(g.nch - kp, rg.u1 - u);
    const int a = run & 1;
    const int n0 = (n + 1 - par) >> 1;   // units of the run at even positions: issuer 0's
    par = (par + n) & 1;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
    ok = ok && __all_sync(0xffffffffu, bwait(&sh.acc_full[a], (run >> 1) & 1, p));
    if (ok) {
      tc_fence_after();
      const uint32_t t = tmem_base + ((uint32_t)(quarter * 32) << 16) + half * 16;
      if (n0 > 0) tmem_ld16_sync(t + a * kTok, v);
      if (n0 < n) {
        float w[16];
        tmem_ld16_sync(t + (a + 2) * kTok, w);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += w[i];
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.acc_empty[a]);
    trace_mark(p, k, 1);
    const int f = grp * kUnitRows + quarter * 32 + lane;
    if (ok && f < g.n_valid) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int tok = half * 16 + i;
        if (tok < p.B) red_add_f32(g.out + tok * g.ldo + f, v[i]);
      }
    }
    trace_mark(p, k, 2);
    ++run;
    u += n;
    ++grp;
    kp = 0;
  }
  sh.ring.skip(rg.u1 - rg.u0);
  return ok;
}

// ---------------------------------------------------------------- attention
template <class T16>
__device__ __forceinline__ void st16(uint8_t* tile, int r, int col, float v) {
  *reinterpret_cast<T16*>(tile + sw_off<16>(r, col >> 3) + (col & 7) * 2) = from_f32<T16>(v);
}

// One K/V tile of kKeys positions for query rows (the group's heads) of one
// warp: S = Q K^T, online softmax in the log2 domain, O += P V.
template <class T16>
__device__ __forceinline__ void attn_tile(const Params& p, uint32_t sq_base, uint8_t* st, int j,
                                          int len, float (&m_r)[2], float (&l_r)[2],
                                          float (&o)[16][4]) {
  const int lane = threadIdx.x % 32;
  const int tq = lane & 3;
  const uint32_t sK = smem_u32(st), sV = sK + 8192;
  const int q_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  // S for 32 keys: four n8 tiles
  float s[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
  {
    const int key = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t qa[4], kb[4], kc[4];
      ldsm_x4(sq_base + sw_off<16>(q_row, 2 * ks + (lane >> 4)), qa);
      ldsm_x4(sK + sw_off<kKeys>(key, 2 * ks + ((lane >> 3) & 1)), kb);
      ldsm_x4(sK + sw_off<kKeys>(key + 16, 2 * ks + ((lane >> 3) & 1)), kc);
      mma16816<T16>(s[0], qa[0], qa[1], qa[2], qa[3], kb[0], kb[1]);
      mma16816<T16>(s[1], qa[0], qa[1], qa[2], qa[3], kb[2], kb[3]);
      mma16816<T16>(s[2], qa[0], qa[1], qa[2], qa[3], kc[0], kc[1]);
      mma16816<T16>(s[3], qa[0], qa[1], qa[2], qa[3], kc[2], kc[3]);
    }
  }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = kKeys * j + nt * 8 + 2 * tq + (e & 1);
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
  uint32_t pa[2][4];
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    float pr[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pr[t][e] = ex2_approx(s[2 * kk + t][e] - m_r[e >> 1]);
        l_r[e >> 1] += pr[t][e];
      }
    pa[kk][0] = pack2<T16>(pr[0][0], pr[0][1]);
    pa[kk][1] = pack2<T16>(pr[0][2], pr[0][3]);
    pa[kk][2] = pack2<T16>(pr[1][0], pr[1][1]);
    pa[kk][3] = pack2<T16>(pr[1][2], pr[1][3]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    o[i][0] *= alpha[0];
    o[i][1] *= alpha[0];
    o[i][2] *= alpha[1];
    o[i][3] *= alpha[1];
  }
  // O += P V over two k16 steps of keys
  {
    const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t vb[4];
        ldsm_x4_t(sV + sw_off<kKeys>(key + 16 * kk, 2 * q + (lane >> 4)), vb);
        mma16816<T16>(o[2 * q], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], vb[0], vb[1]);
        mma16816<T16>(o[2 * q + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], vb[2], vb[3]);
      }
  }
}

// The attention phase of layer l for the CTA's share [f0, f1) of all tiles, in
// rounds. A round takes the rest of the share when that is at most kCons tiles
// (and at most the ring's stages) and touches at most two pairs; then tile t of the
// round goes to warp t, and the two pairs are prepared, computed and combined
// together. Otherwise a round is the rest of the current pair, its tiles taken by
// ring stage (stage index mod kCons).
template <class T16>
__device__ bool consume_attn(const Params& p, Shared& sh, int l, int k) {
  const int warp = threadIdx.x / 32 - 2, lane = threadIdx.x % 32;
  const int tid = threadIdx.x - 64;
  const int gq = lane >> 2, tq = lane & 3;
  Ring& r = sh.ring;
  int f0, f1;
  attn_work(p, blockIdx.x, gridDim.x, f0, f1);
  const int G = p.H / p.Hkv;
  const int qd = p.H * kHd, kvd = p.Hkv * kHd;
  const float* acc_l = p.qkv_acc + (int64_t)(l & 1) * kMaxTok * p.nqkv_pad;
  const float* ss_l = p.ss + (2 * l) * kMaxTok;
  const int npairs = p.B * p.Hkv;
  bool ok = true;
  int f = f0;
  int j0 = 0;
  int bg = f0 < f1 ? pair_at(p, f0, j0) : 0;
  while (f < f1) {
    // ---- the round: pieces (pair, tiles [ja, jb)) of one or two pairs
    int pbg[2], pja[2], pjb[2];
    const int rest = f1 - f;
    pbg[0] = bg;
    pja[0] = j0;
    pjb[0] = min(tiles_of(p, (int)((unsigned)bg / (unsigned)p.Hkv)), j0 + rest);
    const int n0 = pjb[0] - pja[0];
    const bool by_tile = rest <= kCons && rest <= r.n;
    int npc = 1;
    if (by_tile && n0 < rest && bg + 1 < npairs &&
        rest - n0 <= tiles_of(p, (int)((unsigned)(bg + 1) / (unsigned)p.Hkv))) {
      npc = 2;
      pbg[1] = bg + 1;
      pja[1] = 0;
      pjb[1] = rest - n0;
    }
    const int n = npc == 2 ? rest : n0;
    // ---- per piece: the Q tile of the group's query heads (rows >= G zero) and,
    // in the CTA that holds position pos, the new k / v row. Warp w prepares query
    // rows w and w + 8 of each piece; warps 2 pc and 2 pc + 1 also the new k and v
    // of piece pc. All loads of both pieces are issued before any use.
    {
      float av[2][3][4], cv[2][2], sv[2][2], ssb[2];
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        ssb[pc] = 0.f;
#pragma unroll
        for (int rr = 0; rr < 3; ++rr)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) av[pc][rr][jj] = 0.f;
        cv[pc][0] = cv[pc][1] = sv[pc][0] = sv[pc][1] = 0.f;
        if (pc >= npc) continue;
        const int b = (int)((unsigned)pbg[pc] / (unsigned)p.Hkv), g = pbg[pc] - b * p.Hkv;
        const int pos = p.pos[b];
        const bool kv_here = pjb[pc] == tiles_of(p, b) && (warp >> 1) == pc;
        const float* accb = acc_l + (int64_t)b * p.nqkv_pad;
        ssb[pc] = __ldcg(ss_l + b);
        const float* cs = p.cos_tab + (int64_t)pos * (kHd / 2);
        const float* sn = p.sin_tab + (int64_t)pos * (kHd / 2);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          cv[pc][jj] = cs[lane + 32 * jj];
          sv[pc][jj] = sn[lane + 32 * jj];
        }
#pragma unroll
        for (int rr = 0; rr < 3; ++rr) {
          const int hh = warp + 8 * rr;
          const float* src = nullptr;
          if (rr < 2 && hh < G) src = accb + (g * G + hh) * kHd;
          if (rr == 2 && kv_here) src = accb + qd + ((warp & 1) == 0 ? g * kHd : kvd + g * kHd);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) av[pc][rr][jj] = src ? __ldcg(src + lane + 32 * jj) : 0.f;
        }
      }
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        if (pc >= npc) continue;
        const int b = (int)((unsigned)pbg[pc] / (unsigned)p.Hkv), g = pbg[pc] - b * p.Hkv;
        const int pos = p.pos[b];
        const bool kv_here = pjb[pc] == tiles_of(p, b) && (warp >> 1) == pc;
        const float rb = rsqrtf(ssb[pc] / (float)p.d + p.eps);
        uint8_t* sq = sh.sq + pc * 4096;
        uint16_t* kvn = sh.kvnew + pc * 2 * kHd;
#pragma unroll
        for (int rr = 0; rr < 3; ++rr) {
          if (rr == 2 && !kv_here) continue;
          const bool is_v = rr == 2 && (warp & 1) == 1;
          float a4[4], o[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) a4[jj] = av[pc][rr][jj] * rb;
          if (is_v) {
            float amax = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              o[jj] = a4[jj];
              amax = fmaxf(amax, fabsf(o[jj]));
            }
            note_range<T16>(amax, p.status);
          } else {
            float sq2 = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) sq2 += a4[jj] * a4[jj];
            sq2 = warp_sum(sq2);
            const float rn = rsqrtf(sq2 * (1.f / kHd) + p.eps);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const float lo = a4[jj], hi = a4[jj + 2];
              o[jj] = (lo * cv[pc][jj] - hi * sv[pc][jj]) * rn;
              o[jj + 2] = (lo * sv[pc][jj] + hi * cv[pc][jj]) * rn;
            }
          }
          if (rr < 2) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st16<T16>(sq, warp + 8 * rr, lane + 32 * jj, o[jj]);
          } else {
            const int64_t crow =
                (((int64_t)l * p.cache_batch + p.b_off + b) * p.Hkv + g) * p.t_max + pos;
            T16* dstc = static_cast<T16*>(is_v ? p.v_cache : p.k_cache) + crow * kHd;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const T16 v = from_f32<T16>(o[jj]);
              dstc[lane + 32 * jj] = v;
              reinterpret_cast<T16*>(kvn)[(is_v ? kHd : 0) + lane + 32 * jj] = v;
            }
          }
        }
      }
    }
    bar_consumers();
    trace_mark(p, k, 0);
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // One tile of piece pc: wait for its stage, patch the new row into the last
    // tile of the pair, accumulate, release the stage.
    int my_pc = 0;
    auto run_tile = [&](int pc, int j, int st_i, uint32_t par) {
      const int b = (int)((unsigned)pbg[pc] / (unsigned)p.Hkv);
      const int pos = p.pos[b];
      const int last_tile = tiles_of(p, b) - 1;
      ok = ok && __all_sync(0xffffffffu, bwait(&r.full[st_i], par, p));
      uint8_t* st = r.base + (size_t)st_i * kStage;
      if (ok) {
        if (j == last_tile) {
          // the new row from shared memory; V rows past pos zeroed (their p is 0,
          // but a NaN there would still poison the product)
          const int rp = pos - kKeys * last_tile;
          const uint16_t* kvn = sh.kvnew + pc * 2 * kHd;
          for (int i = lane; i < kKeys * 16; i += 32) {
            const int rr = i / 16, c16 = i % 16;
            uint4* kd = reinterpret_cast<uint4*>(st + sw_off<kKeys>(rr, c16));
            uint4* vd = reinterpret_cast<uint4*>(st + 8192 + sw_off<kKeys>(rr, c16));
            if (rr == rp) {
              *kd = reinterpret_cast<const uint4*>(kvn)[c16];
              *vd = reinterpret_cast<const uint4*>(kvn + kHd)[c16];
            } else if (rr > rp) {
              *vd = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          __syncwarp();
        }
        attn_tile<T16>(p, smem_u32(sh.sq + pc * 4096), st, j, pos + 1, m_r, l_r, o);
        // generic writes into the stage are ordered before the next TMA fill
        if (j == last_tile) fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[st_i]);
    };
    if (by_tile) {
      // tile t of the round to warp t: the round's tiles lie in distinct stages,
      // and every earlier position of the ring was consumed before the round
      if (warp < n) {
        int st_i;
        uint32_t par;
        r.ahead(warp, st_i, par);
        my_pc = warp < n0 ? 0 : 1;
        run_tile(my_pc, warp < n0 ? pja[0] + warp : warp - n0, st_i, par);
      }
    } else {
      // Every ring stage belongs to one warp (stage index mod 8), which takes the
      // tiles landing there in order. A warp thus waits on each of its stages'
      // fills one after another and can never reach a fill two ahead of the
      // producer, where the barrier's parity would match an older, completed fill.
      for (int t = 0; t < n; ++t) {
        int st_i;
        uint32_t par;
        r.ahead(t, st_i, par);
        if (st_i % kCons != warp) continue;
        run_tile(0, pja[0] + t, st_i, par);
      }
    }
    r.skip(n);
    trace_mark(p, k, 1);
    // ---- the warps' states against the fixed reference: row sums over the quad,
    // each row's output and sum scaled by 2^(m - kScoreRef) (0 for a warp without
    // keys of the row), summed per piece over its warps through shared memory,
    // then added into the accumulators that all CTAs of the pair share
    float w_r[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
      w_r[h] = ex2_approx(m_r[h] - kScoreRef);
    }
    constexpr int kWs = 16 * kMergeStride + 32;   // floats per warp's merge area
    float* mw = reinterpret_cast<float*>(sh.act) + warp * kWs;
    float* ow = mw + 32;
    if (lane == 0) mw[0] = (float)my_pc;
    if (tq == 0) {
      mw[16 + gq] = l_r[0] * w_r[0];
      mw[16 + gq + 8] = l_r[1] * w_r[1];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = i * 8 + 2 * tq;
      *reinterpret_cast<float2*>(ow + gq * kMergeStride + c) =
          make_float2(o[i][0] * w_r[0], o[i][1] * w_r[0]);
      *reinterpret_cast<float2*>(ow + (gq + 8) * kMergeStride + c) =
          make_float2(o[i][2] * w_r[1], o[i][3] * w_r[1]);
    }
    bar_consumers();
    {
      const float* const mall = reinterpret_cast<const float*>(sh.act);
      const int sl = l & 1;
      for (int e = tid; e < npc * G * (kHd / 4); e += 256) {
        const int pc = e >= G * (kHd / 4) ? 1 : 0;
        const int e1 = e - pc * G * (kHd / 4);
        const int h = e1 / (kHd / 4), i = (e1 % (kHd / 4)) * 4;
        const int b = (int)((unsigned)pbg[pc] / (unsigned)p.Hkv), g = pbg[pc] - b * p.Hkv;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kCons; ++w) {
          if (mall[w * kWs] != (float)pc) continue;
          const float4 ov = *reinterpret_cast<const float4*>(mall + w * kWs + 32 + h * kMergeStride + i);
          v.x += ov.x;
          v.y += ov.y;
          v.z += ov.z;
          v.w += ov.w;
        }
        red_add_f32x4(p.att_num + ((int64_t)sl * kMaxTok + b) * qd + (g * G + h) * kHd + i, v);
      }
      if (tid < npc * G) {
        const int pc = tid >= G ? 1 : 0, h = tid - pc * G;
        const int b = (int)((unsigned)pbg[pc] / (unsigned)p.Hkv), g = pbg[pc] - b * p.Hkv;
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kCons; ++w)
          if (mall[w * kWs] == (float)pc) L += mall[w * kWs + 16 + h];
        red_add_f32(p.att_den + (sl * kMaxTok + b) * p.H + g * G + h, L);
      }
    }
    trace_mark(p, k, 2);
    bar_consumers();
    trace_mark(p, k, 3);
    f += n;
    bg = pbg[npc - 1] + 1;
    j0 = 0;
  }
  return ok;
}

// ---------------------------------------------------------------- small phases
template <class TW>
__device__ void phase_embed(const Params& p) {
  const int tid = threadIdx.x - 64;
  const int gt = blockIdx.x * 256 + tid, gs = gridDim.x * 256;
  for (int i = gt; i < p.B * p.d; i += gs) {
    const int b = (int)((unsigned)i / (unsigned)p.d), k = i - b * p.d;
    int id = p.tokens[b];
    if (id < 0 || id >= p.V) {
      if (k == 0) atomicOr(p.status, ST_BAD_TOKEN);
      id = 0;
    }
    p.x[(int64_t)b * p.d + k] = to_f32(static_cast<const TW*>(p.wte)[(int64_t)id * p.d + k]);
  }
}

// a[0, n) = 0 over the consumer threads of all CTAs (a 16-byte aligned)
__device__ void zero_f32(float* a, int n) {
  const int tid = threadIdx.x - 64;
  const int gt = blockIdx.x * 256 + tid, gs = gridDim.x * 256;
  for (int i = gt * 4; i < n; i += gs * 4) {
    if (i + 4 <= n)
      *reinterpret_cast<float4*>(a + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    else
      for (int k = i; k < n; ++k) a[k] = 0.f;
  }
}

// xn = RMSNorm(x) written as the LM head's B-chunk image: CTA c < kTok writes
// token row c of every chunk (zeros for c >= B).
template <class T16>
__device__ void phase_final_norm(const Params& p) {
  const int tok = blockIdx.x;
  if (tok >= kTok) return;
  const int tid = threadIdx.x - 64;
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
  uint8_t* img = static_cast<uint8_t*>(p.xn_img);
  for (int e = tid; e < p.d / 8; e += 256) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (tok < p.B) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(p.x + (int64_t)tok * p.d + 8 * e));
      const float4 c = __ldcg(reinterpret_cast<const float4*>(p.x + (int64_t)tok * p.d + 8 * e + 4));
      v = make_uint4(pack2<T16>(a.x * r, a.y * r), pack2<T16>(a.z * r, a.w * r),
                     pack2<T16>(c.x * r, c.y * r), pack2<T16>(c.z * r, c.w * r));
    }
    *reinterpret_cast<uint4*>(img + (size_t)(e / 8) * kChunkBytes + bchunk_off(tok, e % 8)) = v;
  }
}

__device__ __forceinline__ uint64_t argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ void phase_argmax(const Params& p) {
  constexpr int kChunk = 2048;
  const int tid = threadIdx.x - 64;
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

// ------------------------------------------------------- sampling mode
// Running softmax state of one token over the vocabulary rows a thread has seen
// (log2 domain: w = 2^((l - m) k), k = log2(e) / temperature) and its greedy best.
struct TokStat {
  float m, s, bv;
  int bi;
};
__device__ __forceinline__ TokStat stat_merge(TokStat a, const TokStat& b, float k) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) {
    a.s = 0.f;
  } else {
    a.s = a.s * ex2_approx((a.m - M) * k) + b.s * ex2_approx((b.m - M) * k);
  }
  a.m = M;
  if (b.bv > a.bv || (b.bv == a.bv && b.bi < a.bi)) {
    a.bv = b.bv;
    a.bi = b.bi;
  }
  return a;
}

// LM head of the sampling mode. The CTA's whole row groups were multiplied into
// their own accumulators; each thread reads its row (vocabulary index f) for 16
// tokens from each of them, writes the logits if asked, and folds them into its
// per-token state. The CTA's states are then merged through shared memory into
// one partial per token in p.lm_part[blockIdx.x]. The accumulators stay in
// tensor memory for the draw.
template <class T16>
__device__ bool consume_lm_sample(const Params& p, Shared& sh, const Gemv& g, int k,
                                  uint32_t tmem_base, int& run) {
  const Range rg = range_of(g);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4, half = (warp - 2) / 4;
  const int tid = threadIdx.x - 64;
  const float kt = p.temp_k;
  TokStat st[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) st[i] = TokStat{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  bool ok = true;
  if (rg.u0 < rg.u1) {
    trace_mark(p, k, 3);
    stage_b<T16>(p, sh, g, rg);
    trace_mark(p, k, 0);
    int grp = rg.g0, rr = 0;
    for (int u = rg.u0; u < rg.u1; u += g.nch, ++grp, ++rr) {
      const int a = run & 1;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
      ok = ok && __all_sync(0xffffffffu, bwait(&sh.acc_full[a], (run >> 1) & 1, p));
      if (ok) {
        tc_fence_after();
        tmem_ld16_sync(tmem_base + ((uint32_t)(quarter * 32) << 16) + kTmemResident + rr * kTok +
                           half * 16,
                       v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[a]);
      ++run;
      const int f = grp * kUnitRows + quarter * 32 + lane;
      if (!ok || f >= g.n_valid) continue;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int tok = half * 16 + i;
        if (p.logits && tok < p.B) p.logits[(int64_t)tok * p.V + f] = v[i];
        if (v[i] > st[i].bv) {   // rows come in increasing f: ties keep the lower index
          st[i].bv = v[i];
          st[i].bi = f;
        }
        if (kt > 0.f) {
          if (v[i] > st[i].m) {
            st[i].s = st[i].s * ex2_approx((st[i].m - v[i]) * kt) + 1.f;
            st[i].m = v[i];
          } else {
            st[i].s += ex2_approx((v[i] - st[i].m) * kt);
          }
        }
      }
    }
    trace_mark(p, k, 1);
  }
  // Every accumulator has been read, so no MMA reads the B chunks any more: the
  // area holds the states, [token][quarter][lane] (token t from the warps of half t / 16).
  bar_consumers();
  TokStat* ts = reinterpret_cast<TokStat*>(sh.act);
#pragma unroll
  for (int i = 0; i < 16; ++i) ts[((half * 16 + i) * 4 + quarter) * 32 + lane] = st[i];
  bar_consumers();
  {
    // thread: token t = tid / 8 merges 16 of the token's 128 states, then 8 lanes merge
    const int t = tid >> 3, part = tid & 7;
    TokStat a{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
    for (int e = part * 16; e < part * 16 + 16; ++e) a = stat_merge(a, ts[t * 128 + e], kt);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      TokStat b;
      b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
      b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
      b.bv = __shfl_xor_sync(0xffffffffu, a.bv, o);
      b.bi = __shfl_xor_sync(0xffffffffu, a.bi, o);
      a = stat_merge(a, b, kt);
    }
    if (part == 0)
      p.lm_part[blockIdx.x * kMaxTok + t] = make_float4(a.m, a.s, a.bv, __int_as_float(a.bi));
  }
  trace_mark(p, k, 2);
  return ok;
}

// The draw. Every CTA merges the partials of all CTAs for each token in the same
// fixed order: the maximum M, then the weights W_c = s_c 2^((m_c - M) k) summed
// one after another, so that CTA c's interval [C_c, C_c + W_c) of [0, Z) is the
// same value in every CTA and the intervals tile [0, Z) exactly. The CTA whose
// interval holds u Z scans its rows of the token in vocabulary order: the
// smallest index whose cumulative weight passes u Z (the last row of nonzero
// weight if rounding leaves it beyond the CTA's rows). Greedy: the best value
// over all partials, lowest index on ties, written by CTA 0.
__device__ void phase_sample(const Params& p, Shared& sh, uint32_t tmem_base) {
  const int tid = threadIdx.x - 64;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;
  const float kt = p.temp_k;
  int* own = reinterpret_cast<int*>(sh.act);                  // [kMaxTok]
  float* resid = reinterpret_cast<float*>(own + kMaxTok);     // [kMaxTok]
  float* mt = resid + kMaxTok;                                // [kMaxTok]
  float* tot = mt + kMaxTok;                                  // [kMaxResidentGroups][4]
  int* found = reinterpret_cast<int*>(tot + 4 * kMaxResidentGroups);   // [1]
  int* lastnz = found + 1;                                    // [4]
  if (tid < kMaxTok) own[tid] = 0;
  bar_consumers();
  if (tid < p.B) {
    const int t = tid;
    float M = -INFINITY, bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = 0; c < (int)gridDim.x; ++c) {
      const float4 e = __ldcg(p.lm_part + c * kMaxTok + t);
      M = fmaxf(M, e.x);
      const int ei = __float_as_int(e.w);
      if (e.z > bv || (e.z == bv && ei < bi)) {
        bv = e.z;
        bi = ei;
      }
    }
    if (!(kt > 0.f)) {
      if (blockIdx.x == 0 && p.argmax_out) p.argmax_out[t] = bi;
    } else {
      float Z = 0.f, C = 0.f, W = 0.f;
      int last = -1;
      for (int c = 0; c < (int)gridDim.x; ++c) {
        const float4 e = __ldcg(p.lm_part + c * kMaxTok + t);
        const float w = e.x == -INFINITY ? 0.f : e.y * ex2_approx((e.x - M) * kt);
        if (c == (int)blockIdx.x) {
          C = Z;
          W = w;
        }
        if (w > 0.f) last = c;
        Z = Z + w;
      }
      const float uu = fminf(fmaxf(__ldcg(p.u + t), 0.f), 0x1.fffffep-1f);
      const float tg = uu * Z;
      int o = (W > 0.f && C <= tg && tg < C + W) ? 1 : 0;
      if (!o && tg >= Z && (int)blockIdx.x == last) o = 2;   // rounded past the total
      own[t] = o;
      resid[t] = o == 2 ? INFINITY : tg - C;
      mt[t] = M;
    }
  }
  bar_consumers();
  if (!(kt > 0.f) || !p.argmax_out) return;
  int g0, g1;
  share(p.vpad / kUnitRows, blockIdx.x, gridDim.x, g0, g1);
  const int ng = g1 - g0;
  for (int t = 0; t < p.B; ++t) {
    if (!own[t]) continue;   // the same decision in every thread (shared memory)
    // warps 2..5 hold the four lane quarters (rows q * 32 + lane of every group)
    const bool scan = warp < 6;
    float incl[kMaxResidentGroups], w[kMaxResidentGroups];
    if (scan) {
      int lnz = -1;
#pragma unroll
      for (int r = 0; r < kMaxResidentGroups; ++r) {
        incl[r] = 0.f;
        w[r] = 0.f;
        if (r >= ng) continue;
        uint32_t raw;
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n"
                     "tcgen05.wait::ld.sync.aligned;\n"
                     : "=r"(raw)
                     : "r"(tmem_base + ((uint32_t)(quarter * 32) << 16) + kTmemResident + r * kTok + t)
                     : "memory");
        const int f = (g0 + r) * kUnitRows + quarter * 32 + lane;
        w[r] = f < p.V ? ex2_approx((__uint_as_float(raw) - mt[t]) * kt) : 0.f;
        float x = w[r];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        incl[r] = x;
        if (lane == 31) tot[r * 4 + quarter] = x;
        if (w[r] > 0.f) lnz = f;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lnz = max(lnz, __shfl_xor_sync(0xffffffffu, lnz, o));
      if (lane == 0) lastnz[quarter] = lnz;
    }
    if (tid == 0) *found = 0;
    bar_consumers();
    if (scan) {
      // base of (group r, quarter q): the totals before it, summed in one fixed order
      const float rs = resid[t];
      float base = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxResidentGroups; ++r) {
        if (r >= ng) break;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q == quarter) {
            const float prev = __shfl_up_sync(0xffffffffu, incl[r], 1);
            const float lo = lane == 0 ? base : base + prev;
            const float hi = base + incl[r];
            if (w[r] > 0.f && lo <= rs && rs < hi) {
              p.argmax_out[t] = (g0 + r) * kUnitRows + quarter * 32 + lane;
              *found = 1;
            }
          }
          base = base + tot[r * 4 + q];
        }
      }
    }
    bar_consumers();
    if (tid == 0 && !*found)
      p.argmax_out[t] = max(max(lastnz[0], lastnz[1]), max(lastnz[2], lastnz[3]));
    bar_consumers();
  }
}

template <class T16, class TW>
__device__ void consumers(const Params& p, Shared& sh, uint32_t tmem_base) {
  int nbar = 0, run = 0;
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 64) p.trace[0] = global_timer_ns();
  // P0: embedding and zeroed accumulators
  phase_embed<TW>(p);
  zero_f32(p.qkv_acc, p.B * p.nqkv_pad);
  zero_f32(p.ss, 2 * p.L * kMaxTok);
  zero_f32(p.att_num, kMaxTok * p.H * kHd);   // layer 0's buffer
  zero_f32(p.att_den, kMaxTok * p.H);
  if (!p.sample) zero_f32(p.logits, p.B * p.V);   // sampling mode stores whole rows
  {
    const int tid = threadIdx.x - 64;
    const int64_t gt = (int64_t)blockIdx.x * 256 + tid;
    if (gt < kMaxTok) {
      p.argmax_key[gt] = 0ull;
      p.argmax_count[gt] = 0u;
    }
  }
  if (!grid_barrier(p, sh, ++nbar)) return;
#pragma unroll 1
  for (int q = 0; q < 5 * p.L + 2; ++q) {
    int ph;
    const int l = phase_layer(q, ph);
    bool ok = true;
    if (l == p.L && ph == 0) {
      phase_final_norm<T16>(p);
    } else if (l < p.L && ph == PH_ATTN) {
      ok = consume_attn<T16>(p, sh, l, nbar + 1);
    } else if (l == p.L && p.sample) {
      ok = consume_lm_sample<T16>(p, sh, gemv_lm(p), nbar + 1, tmem_base, run);
    } else {
      if (l < p.L && ph == PH_QKV) zero_f32(p.hacc, p.B * p.F);
      ok = consume_gemv<T16>(p, sh, l < p.L ? gemv_of(p, l, ph) : gemv_lm(p), nbar + 1, tmem_base, run);
    }
    if (!grid_barrier(p, sh, ++nbar) || !ok) return;
    if (l + 1 < p.L && ph == PH_QKV)
      zero_f32(p.qkv_acc + ((l + 1) & 1) * kMaxTok * p.nqkv_pad, p.B * p.nqkv_pad);
    if (l + 1 < p.L && ph == PH_ATTN) {
      // the next layer's buffer: last read by this layer's predecessor's O phase
      const int sl = (l + 1) & 1;
      zero_f32(p.att_num + (int64_t)sl * kMaxTok * p.H * kHd, p.B * p.H * kHd);
      zero_f32(p.att_den + sl * kMaxTok * p.H, p.B * p.H);
    }
  }
  if (p.sample)
    phase_sample(p, sh, tmem_base);
  else
    phase_argmax(p);
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 64) p.trace[2 * nbar + 1] = global_timer_ns();
}

// ================================================================== kernel
// A failed wait (timeout, or another CTA's abort) never makes a consumer warp
// leave while others may still wait for it at a CTA barrier: inside a phase it
// only skips work; the CTA leaves together at the next grid barrier, whose
// result every consumer thread shares. All roles then meet at the final CTA
// barrier, after which warp 1 frees the tensor memory.
template <class T16, class TW>
__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ Params p) {
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
  q += p.act_bytes;
  sh.sq = q;
  q += 8192;   // Q tiles of up to two pairs
  sh.kvnew = reinterpret_cast<uint16_t*>(q);
  q += 1024;   // new K and V rows of up to two pairs
  sh.ring.full = reinterpret_cast<uint64_t*>(q);
  sh.ring.empty = sh.ring.full + p.stages;
  sh.acc_full = sh.ring.empty + p.stages;
  sh.acc_empty = sh.acc_full + 2;
  sh.b_full = sh.acc_empty + 2;
  sh.fin = sh.b_full + 1;
  sh.tmem_slot = reinterpret_cast<uint32_t*>(sh.fin + 1);
  sh.flag = reinterpret_cast<volatile int*>(sh.tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sh.ring.full[s], 1);
      mbar_init(&sh.ring.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.acc_full[a], 2);   // one commit per MMA issuer
      mbar_init(&sh.acc_empty[a], kCons);
    }
    mbar_init(sh.b_full, kCons);
    mbar_init(sh.fin, 2);
    sh.flag[2] = 1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sh.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sh.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      producer(p, sh.ring, &tmK, &tmV);
    }
  } else if (warp == 1 || warp == 2 + kCons) {
    if (lane == 0) mma_role<T16>(p, sh, sh.ring, tmem_base, warp == 1 ? 0 : 1);
  } else {
    consumers<T16, TW>(p, sh, tmem_base);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ===================================================================== host
// Packs rows [0, Npad) of W = [W0; W1; W2] (row-major [N, K], rows split at s0,
// s1; rows >= N zero) into 16 KB units of 128 rows x 64 columns: unit (grp, c)
// at ((grp * K/64 + c) * 16384); inside it row r's 128 bytes at r * 128 with
// 16-byte chunk j (columns c*64 + 8j .. + 7) at position j XOR (r % 8): the
// 128-byte-swizzled K-major layout, so a 1-D copy to a 1024-byte aligned stage
// gives the tensor core's A operand as it is.
template <class T16>
__global__ void pack_kernel(const T16* __restrict__ w0, const T16* __restrict__ w1,
                            const T16* __restrict__ w2, int s0, int s1, int N, int K,
                            int64_t n_entries, uint4* __restrict__ out) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_entries) return;
  const int pj = (int)(e & 7);            // physical 16-byte position in the row
  const int r = (int)((e >> 3) & 127);    // row of the unit
  const int64_t unit = e >> 10;
  const int nch = K / kUnitCols;
  const int grp = (int)(unit / nch), c = (int)(unit % nch);
  const int j = pj ^ (r & 7);             // logical chunk stored there
  const int row = grp * kUnitRows + r;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row < N) {
    const T16* src = row < s0 ? w0 + (int64_t)row * K
                              : row < s1 ? w1 + (int64_t)(row - s0) * K : w2 + (int64_t)(row - s1) * K;
    v = *reinterpret_cast<const uint4*>(src + c * kUnitCols + 8 * j);
  }
  out[e] = v;
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
  lo.xn_img_bytes = (int64_t)(d / kUnitCols) * kChunkBytes;
  return lo;
}

// Shared memory of a launch: the ring, the B-chunk / merge area, the Q tile,
// the new K/V row, barriers and flags. The B area holds the most chunks any
// CTA's range of any projection needs, and at least every chunk of d_model.
static int b_slots_needed(int d, int H, int F, int nqkv_pad, int vpad, int P) {
  auto need = [&](int64_t units, int nch) {
    const int64_t per = (units + P - 1) / P;
    return (int)std::min<int64_t>(per, nch);
  };
  const int qd = H * kHd;
  int n = need((int64_t)(nqkv_pad / kUnitRows) * (d / kUnitCols), d / kUnitCols);
  n = std::max(n, need((int64_t)(d / kUnitRows) * (qd / kUnitCols), qd / kUnitCols));
  n = std::max(n, need((int64_t)(F / kUnitRows) * (d / kUnitCols), d / kUnitCols));
  n = std::max(n, need((int64_t)(d / kUnitRows) * (F / kUnitCols), F / kUnitCols));
  // the LM head: every chunk of d (a CTA that owns whole row groups in sampling
  // mode stages all of them, whatever the vocabulary)
  n = std::max(n, d / kUnitCols);
  (void)vpad;
  return n;
}

static size_t smem_bytes(int act, int* stages) {
  const int fixed = 1024 /*align*/ + 8192 + 1024 + 256;
  const int limit = 232448 - 1024;   // dynamic part; static shared memory is small
  int st = (limit - fixed - act) / (kStage + 16);
  if (st > 16) st = 16;
  st &= ~1;   // even: each stage belongs to one of the two MMA issuers
  *stages = st;
  return (size_t)st * kStage + act + fixed + 16 * st;
}

bool supported(int d, int H, int Hkv, int F, int hd, int V, int P) {
  if (!(hd == kHd && H % Hkv == 0 && H / Hkv <= 16 && d % kUnitRows == 0 && F % kUnitRows == 0))
    return false;
  // work ranges are computed in 32 bits: units * P must stay below 2^31
  const int64_t units_max = std::max<int64_t>(
      std::max<int64_t>(round_up(V, kUnitRows) / kUnitRows * (d / kUnitCols),
                        (int64_t)(F / kUnitRows) * (d / kUnitCols)),
      (int64_t)(d / kUnitRows) * (F / kUnitCols));
  if (units_max * (P + 1) >= (int64_t(1) << 31)) return false;
  const int nqkv = (H + 2 * Hkv) * kHd;
  const int act = std::max(b_slots_needed(d, H, F, (int)round_up(nqkv, kUnitRows),
                                          (int)round_up(V, kUnitRows), P) * kChunkBytes,
                           kMergeBytes);
  int st = 0;
  smem_bytes(act, &st);
  return st >= 4;
}

int plan_attention(Params& p, int P) {
  const int pairs = p.B * p.Hkv;
  int64_t total = 0;
  for (int b = 0; b < p.B; ++b) {
    if (total >= (int64_t(1) << 31)) return -1;
    p.tile_pre[b] = (int)total;
    total += (int64_t)tiles_of(p, b) * p.Hkv;
  }
  if (total * (P + 1) >= (int64_t(1) << 31)) return -1;
  p.tile_pre[p.B] = (int)total;
  p.attn_total = (int)total;
  // Even shares of all tiles when no share exceeds kCons tiles and none can span
  // more than two pairs (every pair at least the largest share minus one tiles):
  // each CTA then computes its tiles in one round, one per warp. Otherwise, with
  // no more pairs than CTAs, per-pair CTA blocks (one pair per CTA).
  int min_tiles = INT_MAX;
  for (int b = 0; b < p.B; ++b) min_tiles = std::min(min_tiles, tiles_of(p, b));
  const int64_t largest = (total + P - 1) / P;
  const bool even = largest <= kCons && min_tiles >= largest - 1;
  p.attn_blocks = (!even && pairs <= P && P <= kMaxAttnBlocks) ? 1 : 0;
  if (p.attn_blocks) {
    // every pair one CTA, the other P - pairs CTAs in proportion to its tiles
    for (int bg = 0; bg <= pairs; ++bg) {
      const int64_t t0 = bg == pairs ? total : tile0_of(p, bg);
      p.pair_c0[bg] = (unsigned short)(bg + (int64_t)(P - pairs) * t0 / total);
    }
  }
  return 1;
}

template <class T16, class TW>
static nc_status launch_t(const CUtensorMap& tk, const CUtensorMap& tv, Params p, int sms,
                          size_t smem, cudaStream_t s) {
  auto kern = decode_step_kernel<T16, TW>;
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

nc_status launch_step(const CUtensorMap& tk, const CUtensorMap& tv, Params p, bool half,
                      nc_dtype wdt, int sms, cudaStream_t s) {
  if ((int64_t)p.attn_total * (sms + 1) >= (int64_t(1) << 31)) {
    set_last_error("decode step: attention work of %d sequences is too large", p.B);
    return NC_ERR_UNSUPPORTED;
  }
  const int act = (int)round_up(std::max(b_slots_needed(p.d, p.H, p.F, p.nqkv_pad, p.vpad, sms) *
                                             kChunkBytes,
                                         kMergeBytes),
                                1024);
  int stages = 0;
  const size_t smem = smem_bytes(act, &stages);
  if (stages < 4) {
    set_last_error("decode step: shared memory too small for the ring (%d stages)", stages);
    return NC_ERR_UNSUPPORTED;
  }
  p.stages = stages;
  p.act_bytes = act;
  if (half) {
    if (wdt == NC_BF16) return launch_t<f16, bf16>(tk, tv, p, sms, smem, s);
    if (wdt == NC_F16) return launch_t<f16, f16>(tk, tv, p, sms, smem, s);
    return launch_t<f16, float>(tk, tv, p, sms, smem, s);
  }
  if (wdt == NC_BF16) return launch_t<bf16, bf16>(tk, tv, p, sms, smem, s);
  if (wdt == NC_F16) return launch_t<bf16, f16>(tk, tv, p, sms, smem, s);
  return launch_t<bf16, float>(tk, tv, p, sms, smem, s);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D view [rows, 128] of a 16-bit KV array, boxes of kKeys rows x 64 columns
// with the 128-byte swizzle (the layout the attention phase reads).
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
  cuuint32_t box[2] = {64, (cuuint32_t)kKeys};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dec
}  // namespace nc
