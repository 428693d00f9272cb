// Tensor-core (bf16) part of the forward pass: tcgen05 GEMMs with fused
// epilogues, and prefill attention.
#pragma once
#include "nc_internal.h"

namespace nc {

constexpr int kMaxSplits = 16;      // split-K factor limit of the small-M projections
constexpr int kSwapMaxRows = 128;   // M <= this runs weight-stationary (swap-AB) GEMMs

struct TcModel;

// Weight pointers are in cfg.act_dtype (the caller converts first if needed).
nc_status tc_create(const nc_config& cfg, const void* lm_head, const void* const* wq,
                    const void* const* wk, const void* const* wv, const void* const* wo,
                    const void* const* w_fc, const void* const* w_proj, void* xn, void* att,
                    void* h, void* xnl, size_t max_rows, uint32_t* status, TcModel** out);
void tc_destroy(TcModel* t);

// Q/K/V projections of rows xn[M, d] with RoPE, QK norm and the scatter to q and
// the KV cache fused in (or applied by a finishing kernel for small M).
nc_status tc_qkv(TcModel* t, int layer, int64_t M, const RowMap& rm, const QkvDst& dst,
                 float* part, cudaStream_t s);
// x += att W_o^T
nc_status tc_out_proj(TcModel* t, int layer, int64_t M, float* x, float* part, cudaStream_t s);
// h = relu(xn W_fc^T)^2
nc_status tc_fc(TcModel* t, int layer, int64_t M, float* part, cudaStream_t s);
// x += h W_proj^T
nc_status tc_proj(TcModel* t, int layer, int64_t M, float* x, float* part, cudaStream_t s);
// logits[M, V] = xn lm_head^T (xn is the model's xn or xnl buffer)
nc_status tc_lm_head(TcModel* t, const void* xn, int64_t M, float* logits, float* part,
                     cudaStream_t s);
// The same product reduced per row and block of 256 columns, no logits stored:
// part[nb * M + r] = (max, sum exp(z - max)) over block nb of row r's logits, and
// zt[r] = the logit of column targets[r] (written where 0 <= targets[r] < V).
// part holds lm_loss_blocks(V) * M pairs.
int lm_loss_blocks(int vocab);
nc_status tc_lm_loss(TcModel* t, const void* xn, int64_t M, const int32_t* targets, float2* part,
                     float* zt, cudaStream_t s);
// Causal attention over q [B, H, T, 128], cache k/v [B, Hkv, t_max, 128] -> o [B, T, H*128].
nc_status tc_attention_prefill(const void* q, const void* k, const void* v, void* o, int B, int H,
                               int Hkv, int T, int t_max, nc_dtype dt, cudaStream_t s);
// The same attention on tcgen05 (TMEM scores and output, TMA-fed K/V rings), for
// queries at absolute positions pos0 .. pos0 + T - 1 (q row i is position pos0 + i)
// over keys 0 .. pos0 + T - 1. K/V of layer `layer` are k/v + layer * layer_stride
// elements ([B_cache, Hkv, t_max, 128] each, sequences 0..B-1 and rows
// < pos0 + T read). status: device word for bounded-wait timeouts (NULL: a
// library-wide word). NC_ERR_INVALID_ARG if pos0 < 0 or pos0 + T > t_max.
nc_status tc_attention_prefill_tc(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int T, int pos0, int t_max, int n_layers,
                                  int64_t layer_stride, int layer, nc_dtype dt, uint32_t* status,
                                  cudaStream_t s);
// fp8 (E4M3) projection variant: row-wise quantisation and the scaled product
nc_status quantize_e4m3(const void* x, nc_dtype dt, int64_t rows, int cols, uint8_t* q, float* scale,
                        cudaStream_t s);
size_t gemv_e4m3_scratch_bytes(int N, int K, int B);
nc_status gemv_e4m3(const uint8_t* wq, const float* w_scale, int N, int K, const float* x, int B,
                    float* y, void* scratch, cudaStream_t s);
// The cross-entropy reduction of C = A B^T against targets (single-step entry
// point): part and zt as tc_lm_loss, for lm_loss_blocks(N) blocks.
nc_status tc_cross_entropy(const void* A, const void* B, const int32_t* targets, int M, int N,
                           int K, nc_dtype dt, float2* part, float* zt, cudaStream_t s);
// C[M, N] = A[M, K] B[N, K]^T, fp32 out (single-step entry point).
nc_status tc_gemm_f32out(const void* A, const void* B, float* C, int M, int N, int K, nc_dtype dt,
                         cudaStream_t s);


}  // namespace nc
