// Tensor-core (bf16) part of the forward pass: tcgen05 GEMMs with fused
// epilogues, and prefill attention.
#pragma once
#include "nc_internal.h"

namespace nc {

constexpr int kMaxSplits = 16;      // split-K factor limit of the small-M projections
constexpr int kSwapMaxRows = 128;   // M <= this runs weight-stationary (swap-AB) GEMMs

struct TcModel;

nc_status tc_create(const nc_config& cfg, const void* wte, const void* lm_head,
                    const void* const* wq, const void* const* wk, const void* const* wv,
                    const void* const* wo, const void* const* w_fc, const void* const* w_proj,
                    void* xn, void* att, void* h, void* xnl, size_t max_rows, uint32_t* status,
                    TcModel** out);
void tc_destroy(TcModel* t);

// Q/K/V projections of rows xn[M, d] with RoPE, QK norm and the scatter to q and
// the KV cache fused in (or applied by a finishing kernel for small M).
nc_status tc_qkv(TcModel* t, int layer, int64_t M, const RowMap& rm, const QkvDst& dst,
                 float* part, cudaStream_t s);
// x += att W_o^T
nc_status tc_out_proj(TcModel* t, int layer, int64_t M, float* x, float* part, cudaStream_t s);
// x += relu(xn W_fc^T)^2 W_proj^T
nc_status tc_mlp(TcModel* t, int layer, int64_t M, float* x, float* part, cudaStream_t s);
// logits[M, V] = xn lm_head^T (xn is the model's xn or xnl buffer)
nc_status tc_lm_head(TcModel* t, const void* xn, int64_t M, float* logits, float* part,
                     cudaStream_t s);
// Causal attention; t may be NULL (single-step entry point).
nc_status tc_attention_prefill(TcModel* t, const void* q, const void* k, const void* v, void* o,
                               int B, int H, int Hkv, int T, int t_max, cudaStream_t s);
// C[M, N] = A[M, K] B[N, K]^T, fp32 out (single-step entry point).
nc_status tc_gemm_f32out(const void* A, const void* B, float* C, int M, int N, int K,
                         cudaStream_t s);

}  // namespace nc
