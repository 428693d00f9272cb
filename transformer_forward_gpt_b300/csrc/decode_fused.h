// Host interface of the persistent single-launch decode step (decode_fused.cu).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "nc_internal.h"

namespace nc {
namespace dec {

constexpr int kMaxTok = 32;   // sequences per launch (larger batches run in chunks)

// Byte layout of the packed decode weights: per layer [QKV | O | FC | PROJ],
// then the LM head; each matrix in 16 KB units of 128 rows x 64 columns. The
// final norm is kept as an image of the LM head's B operand: per 64-column
// chunk, kMaxTok token rows of 128 bytes.
struct Layout {
  int nqkv, nqkv_pad, vpad;
  int64_t off_o, off_fc, off_proj, layer_bytes, total_bytes;
  int64_t xn_img_bytes;
};

struct PackSrc {
  int L, d, H, Hkv, F, V;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* wfc;
  const void* const* wproj;
  const void* lm;
};

// Attention work of a launch is cut into tiles of 32 positions per (sequence,
// KV head) pair. With no more pairs than CTAs, pair bg owns the CTA block
// [pair_c0[bg], pair_c0[bg + 1]) and spreads its tiles over it; otherwise the
// tiles of all pairs, concatenated, are shared evenly.
constexpr int kMaxAttnBlocks = 256;

struct Params {
  int B, b_off, cache_batch, t_max;
  int pos[kMaxTok];           // position of each sequence's new token (its cache length)
  int tile_pre[kMaxTok + 1];  // attention tiles of the pairs of sequences 0..b-1 (all KV heads)
  int attn_total;             // attention tiles of all pairs
  int attn_blocks;            // 1: per-pair CTA blocks (pair_c0); 0: tiles shared evenly
  unsigned short pair_c0[kMaxAttnBlocks + 1];
  int L, d, H, Hkv, F, V, vpad, nqkv, nqkv_pad;
  int stages, act_bytes;
  float eps, scale_log2;
  int64_t layer_bytes, off_o, off_fc, off_proj;
  const int32_t* tokens;      // [B]
  int32_t* argmax_out;        // [B] or null
  const void* wte;            // [V, d] in the model's weight type
  const uint8_t* wpack;
  const float* cos_tab;
  const float* sin_tab;
  void* k_cache;              // K of layer 0 (all layers follow), 16-bit
  void* v_cache;
  float* x;                   // [kMaxTok, d] residual
  float* qkv_acc;             // [2][kMaxTok][nqkv_pad]
  float* hacc;                // [kMaxTok][F]
  float* ss;                  // [2 L][kMaxTok]
  void* xn_img;               // final norm, B-chunk image [d/64][kMaxTok][128 B]
  float* logits;              // [B][V]; in sampling mode optional (NULL: never written)
  // Sampling mode: the LM head gives every CTA whole row groups of the vocabulary,
  // keeps their logits in tensor memory, and the step ends with a draw from
  // softmax(logits / temperature) (the greedy index when temp_k is 0) instead of
  // a pass over the logits in memory.
  int sample;
  float temp_k;               // log2(e) / temperature, 0 for the greedy index
  const float* u;             // [B] uniforms in [0, 1), one per sequence
  float4* lm_part;            // [gridDim][kMaxTok] per CTA: max, exp-sum, best value, best index
  // Attention output of a layer as sums over the CTAs that share a (sequence, KV
  // head) pair: numerators sum_c 2^(m_c - ref) o_c and denominators
  // sum_c 2^(m_c - ref) l_c of each CTA's softmax state (max m_c, sum l_c,
  // unnormalised output o_c) against one fixed reference. Two buffers, by layer
  // parity; each is zeroed a layer ahead of its use.
  float* att_num;             // [2][kMaxTok][H * 128]
  float* att_den;             // [2][kMaxTok][H]
  unsigned long long* argmax_key;   // [kMaxTok]
  unsigned int* argmax_count;       // [kMaxTok]
  unsigned long long* bar_counter;  // grid barrier arrivals (monotonic)
  unsigned long long bar_base;      // its value when this launch starts
  uint32_t* status;
  uint32_t* abort;
  // optional: %globaltimer of CTA 0 at start, at each grid barrier (arrival,
  // exit) and at the end (2 * nbar + 2 entries), then 4 marks inside each phase
  unsigned long long* trace;
  int nbar;                   // grid barriers of this launch
};

Layout layout_of(int L, int d, int H, int Hkv, int F, int V);
int64_t packed_bytes(int N, int K);
// Whether the persistent step has a configuration for this shape on P SMs.
bool supported(int d, int H, int Hkv, int F, int hd, int V, int P);
nc_status pack_weights(const PackSrc& src, bool half, uint8_t* out, cudaStream_t s);
// Fills p.tile_pre, p.attn_total, p.attn_blocks and p.pair_c0 from p.pos, p.B,
// p.Hkv for P CTAs; returns 1, or -1 if the work is too large for 32-bit indices.
int plan_attention(Params& p, int P);
// TMA view of a KV array (all layers) as [rows, 128] 16-bit values.
bool make_cache_map(CUtensorMap* map, void* base, uint64_t rows, bool half);
// Vocabulary row groups a CTA may keep in tensor memory in sampling mode.
constexpr int kMaxResidentGroups = 6;
// Grid barriers one launch passes (its arrivals are that times the grid size).
inline int barriers_per_step(int L) { return 5 * L + 3; }
// CTAs whose barrier arrival and exit times a trace records.
constexpr int kTraceCtas = 256;
// Entries of a full trace: CTA 0's barrier times, 6 marks per phase, then per
// barrier and CTA (up to kTraceCtas) its arrival and exit time.
inline int trace_entries(int L) {
  return 8 * barriers_per_step(L) + 2 + 2 * kTraceCtas * barriers_per_step(L);
}
// Enqueues one step for p.B <= kMaxTok sequences on `sms` CTAs (cooperative launch).
nc_status launch_step(const CUtensorMap& tk, const CUtensorMap& tv, Params p, bool half,
                      nc_dtype wdt, int sms, cudaStream_t s);

}  // namespace dec
}  // namespace nc
