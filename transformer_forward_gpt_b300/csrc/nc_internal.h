// Internal launch interface shared by the .cu files of the library (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nc.h"

namespace nc {

// Process-wide count of kernel launches made by the library (measurement only).
void count_launches(int n);
// Sets the thread-local text nc_last_error() returns.
void set_last_error(const char* fmt, ...);
// Raises the dynamic shared-memory limit of kernel `func` to at least `bytes` on
// the current device. The attribute belongs to one device, so the sizes already
// set are remembered per (kernel, device); concurrent callers are serialised.
// Returns false if the runtime refuses.
bool ensure_dyn_smem(const void* func, size_t bytes);

// Where the rows of a projection output go (prefill: rows = B*T tokens of B
// sequences starting at position pos0 = 0; decode: rows = B, one per sequence, at
// position pos0 = pos).
struct RowMap {
  int32_t rows_per_seq;   // T (prefill) or 1 (decode)
  int32_t pos0;           // absolute position of row 0 of each sequence
};

// Destinations of the Q/K/V projection epilogue (RoPE + QK norm + scatter).
struct QkvDst {
  void* q;                // [B, H, rows_per_seq, hd]
  void* k_cache;          // [B_cache, Hkv, t_max, hd] of this layer
  void* v_cache;
  int32_t H, Hkv, hd, t_max;
  const float* cos_tab;   // [max_seq, hd/2]
  const float* sin_tab;
  float eps;
  const float* cos_t;     // the same tables position-minor: [hd/2, max_seq]
  const float* sin_t;
  int32_t tab_ld;         // max_seq
  uint32_t* status;       // device status word (fp16 range of the V rows), or NULL
};

// ---- CUDA-core kernels (simt.cu)
void launch_embed_norm(const int32_t* tok, const void* wte, nc_dtype wdt, float* x, void* xn,
                       nc_dtype adt, int64_t M, int d, int vocab, float eps, uint32_t* status,
                       cudaStream_t s);
void launch_rmsnorm(const float* x, void* y, nc_dtype ydt, int64_t M, int d, float eps,
                    cudaStream_t s);
void launch_gemm_simt(const void* A, const void* B, float* C, int64_t M, int N, int K,
                      int64_t ldc, nc_dtype dt, cudaStream_t s);
// out-of-place reductions of split-K partials part[split][M][N] (split stride
// = M*N) followed by one epilogue each
void launch_qkv_post(const float* part, int n_split, int64_t M, const RowMap& rm,
                     const QkvDst& dst, nc_dtype dt, cudaStream_t s);
void launch_residual_finish(const float* part, int n_split, float* x, int64_t M, int N,
                            void* xn_out, nc_dtype dt, float eps, cudaStream_t s);
void launch_relu2_finish(const float* part, int n_split, void* h, int64_t M, int N, nc_dtype dt,
                         uint32_t* status, cudaStream_t s);
void launch_sum_splits(const float* part, int n_split, float* out, int64_t M, int N, int64_t ldo,
                       cudaStream_t s);
void launch_attention_prefill_simt(const void* q, const void* k, const void* v, void* o, int B,
                                   int H, int Hkv, int T, int t_max, int hd, nc_dtype dt,
                                   cudaStream_t s);
// Decode attention: the key range [0, len) of each (sequence, KV head) is cut into
// n_split ranges of tiles_per_split 64-key tiles; each range writes one partial
// (m, l, o[hd]) per query head to scratch[((b*H + h)*n_split + split)*(hd + 2)].
void decode_attention_plan(int len, int bg, int* tiles_per_split, int* n_split);
size_t decode_attention_scratch_bytes(int B, int H, int Hkv, int len, int hd);
bool decode_attention_mma_ok(int H, int Hkv, int hd, nc_dtype dt);
// Picks the tensor-core kernel when it applies, else the CUDA-core one; then merges.
void launch_attention_decode(const void* q, const void* k, const void* v, void* o, int B, int H,
                             int Hkv, int len, int t_max, int hd, nc_dtype dt, float* scratch,
                             cudaStream_t s);
void launch_attention_decode_mma(const void* q, const void* k, const void* v, void* o, int B,
                                 int H, int Hkv, int len, int t_max, nc_dtype dt, float* scratch,
                                 cudaStream_t s);
void launch_attention_decode_simt(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int len, int t_max, int hd, nc_dtype dt,
                                  float* scratch, int n_split, cudaStream_t s);
void launch_attention_combine(const float* scratch, void* o, int BH, int hd, int n_split,
                              nc_dtype dt, cudaStream_t s);
// dst[i] = src[i] converted between number formats (weight copies).
void launch_convert16(const void* src, nc_dtype from, void* dst, nc_dtype to, int64_t n,
                      cudaStream_t s);
void launch_argmax(const float* x, int rows, int n, int32_t* out, cudaStream_t s);
// ---- next-token loss (loss.cu): loss[r] = log sum_nb s_nb exp(m_nb - M_r) + M_r
// - zt[r] from the LM head's per-block softmax partials part[nb * M + r]; rows
// whose target is outside [0, V) get 0 and are not counted (targets >= V also set
// ST_BAD_TOKEN in status, if not NULL); mean = sum of the counted losses / their number
// (NaN if none), summed in a fixed order.
void launch_ce_finish(const float2* part, int nblk, const float* zt, const int32_t* targets,
                      int V, int64_t M, float* loss, float* mean, uint32_t* status,
                      cudaStream_t s);

// ---- temperature sampling (sample.cu)
void launch_sample(const float* logits, int B, int V, float temperature, const float* u,
                   int32_t* out, cudaStream_t s);
void launch_gather_rows(const float* x, float* y, int B, int T, int d, cudaStream_t s);

}  // namespace nc
