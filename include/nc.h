/*
 * nc.h -- C ABI of the B300 (sm_103a) forward pass of a nanochat-style GPT.
 *
 * The model is the decoder-only transformer the pages describe: token
 * embedding; per block RMSNorm (no gain), separate Q/K/V projections, rotary
 * embedding on precomputed cos/sin tables, QK RMS-norm, causal multi-/grouped-
 * query attention, output projection + residual, RMSNorm, ReLU^2 MLP +
 * residual; final RMSNorm and an untied LM head. Sources, by page and section:
 *   - 復刻 ChatGPT 有多難？ (jxzklqfsx.com), section 為什么可以訓練如此之快:
 *     own RoPE that splits a vector into two halves and rotates them; Q, K, V as
 *     separate linear layers; ReLU2 activation; cos/sin precomputed and kept in
 *     GPU memory; KV cache with a branch on whether the cache exists; dense MLP.
 *   - 8000行手写代码！nanochat (hongdingcd.com): dense Transformer, rotary
 *     embedding, QK normalisation; MQA and the KV cache for single-GPU inference.
 *   - CSDN nanochat article (wap.jaobe.com), inference paragraph: an Engine with
 *     a KV cache and the two phases prefill and decode.
 *   - Microgpt summary (telegra.ph), sections 模型参数 and 核心架构: RMSNorm
 *     instead of LayerNorm, no biases, matrices only (embedding, attention, MLP,
 *     final output projection), softmax, attention over the current and earlier
 *     positions, two-layer MLP, residual connections, KV cache; section 推理:
 *     generation feeds the sampled token back, one position at a time.
 *
 * Conventions shared by every entry point:
 *   - Every matrix is row-major [out, in]: y = x W^T. Head h of the Q projection
 *     owns output rows [h*hd, (h+1)*hd); KV head g likewise.
 *   - "dev" pointers are CUDA device pointers on the current device; "host"
 *     pointers are host memory (pinned memory lets copies overlap).
 *   - Device pointers handed to the library must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it; results are ready once the stream
 *     is synchronised. A model and its caches are used from one stream at a time.
 *   - Every call returns an nc_status and never throws. Errors found on the host
 *     (bad sizes, null or misaligned pointers, positions out of range) return
 *     at once and enqueue nothing. Errors found on the device (a token id out of
 *     [0, vocab), an internal wait that timed out) latch in a per-model status
 *     word that nc_model_check() reads. nc_last_error() gives a thread-local
 *     text for the last failure.
 */
#ifndef NC_H_
#define NC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NC_API __attribute__((visibility("default")))

typedef enum {
    NC_OK = 0,
    NC_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, size or position out of range */
    NC_ERR_UNSUPPORTED = 2,     /* shape the library has no kernel for */
    NC_ERR_OOM = 3,             /* device allocation failed */
    NC_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed */
    NC_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait ran out (device status word) */
    NC_ERR_BOUNDS = 6,          /* a token id outside [0, vocab) was seen (device status word);
                                   the kernel used row 0 in its place (an input token) or
                                   left the row out (a loss target >= vocab) */
    NC_ERR_RANGE = 7            /* a value stored in fp16 (act_dtype NC_F16) was too large for
                                   it and became +-inf (device status word): the V rows of the
                                   KV cache, the ReLU^2 activations, or the decode step's
                                   un-normalised residual; NC_BF16 has fp32's range */
} nc_status;

typedef enum { NC_F32 = 0, NC_BF16 = 1, NC_F16 = 2 } nc_dtype;

/* Model shape and number formats.
 *   dtype      storage type of the caller's weights: NC_F32, NC_BF16 or NC_F16.
 *   act_dtype  16-bit type of the tensor-core path (ignored for NC_F32 weights,
 *              which run an fp32 CUDA-core path for small shapes): the format of
 *              the GEMM operands, the normalised activations, Q and the KV cache.
 *              NC_F16 keeps 3 more mantissa bits than NC_BF16 at the same speed
 *              and width; with bf16 rounding at every GEMM input the logits drift
 *              ~0.03-0.04 x RMS (max) from exact arithmetic, with fp16 ~0.005.
 *              When act_dtype differs from dtype the model keeps its own converted
 *              copy of the projection and LM-head weights.
 * The tensor-core path needs head_dim == 128, d_model % 64 == 0, d_mlp % 64 == 0;
 * the fp32 path head_dim <= 128 and even. Residual stream and logits are fp32.
 * max_batch * max_seq bounds the tokens of one prefill call and max_seq bounds
 * every position (cos/sin tables are built for max_seq positions). */
typedef struct {
    int32_t vocab, d_model, n_layer, n_head, n_kv_head, head_dim, d_mlp;
    float rope_base;   /* theta(t, i) = t * rope_base^(-2 i / head_dim) */
    float rms_eps;     /* x / sqrt(mean(x^2) + rms_eps) */
    int32_t max_seq, max_batch;
    nc_dtype dtype;
    nc_dtype act_dtype;
} nc_config;

/* Weights: device pointers in cfg.dtype, row-major [out, in]. Borrowed: the
 * caller keeps them alive and unchanged for the model's lifetime (wte always;
 * the others unless the model converted them at create). The per-layer
 * members are HOST arrays of n_layer device pointers (read during create only).
 *   wte [vocab, d]      lm_head [vocab, d]       (untied)
 *   wq [H*hd, d]  wk [Hkv*hd, d]  wv [Hkv*hd, d]  wo [d, H*hd]
 *   w_fc [d_mlp, d]  w_proj [d, d_mlp]                                        */
typedef struct {
    const void* wte;
    const void* lm_head;
    const void* const* wq;
    const void* const* wk;
    const void* const* wv;
    const void* const* wo;
    const void* const* w_fc;
    const void* const* w_proj;
} nc_weights;

typedef struct nc_model nc_model;
typedef struct nc_kv_cache nc_kv_cache;

NC_API const char* nc_version(void);
NC_API const char* nc_status_string(nc_status s);
/* Thread-local description of the last failing call ("" if none). */
NC_API const char* nc_last_error(void);

/* Number of weight values of a shape: 2*vocab*d + n_layer*(per-layer matrices). */
NC_API int64_t nc_param_count(const nc_config* cfg);

/* The model's parameters are the matrices the Microgpt summary lists in section
 * 模型参数 (token embedding, the attention and MLP matrices of every layer, and
 * the final output projection; no biases, no norm gains); the cos/sin tables are
 * the precomputed rotary embedding of 復刻 ChatGPT 有多難？ (jxzklqfsx.com),
 * section 為什么可以訓練如此之快, kept in GPU memory.
 * Validates cfg, builds the cos/sin tables (computed in fp64 on the host, stored
 * fp32 on the device), allocates the workspace for max_batch*max_seq tokens and
 * the device status word, and builds the TMA descriptors of the weights. Uses the
 * current CUDA device. On failure *out is NULL and nothing is leaked. */
NC_API nc_status nc_model_create(const nc_config* cfg, const nc_weights* w, nc_model** out);
NC_API void nc_model_destroy(nc_model* m);

/* Bytes of a KV cache: 2 (K and V) * n_layer * batch * n_kv_head * t_max * head_dim
 * * sizeof(activation type), plus 256 bytes of header. Layout of K (and V):
 * [n_layer][batch][n_kv_head][t_max][head_dim]; K is stored after RoPE and QK
 * norm, V as projected. */
NC_API size_t nc_kv_cache_bytes(const nc_config* cfg, int32_t batch, int32_t t_max);

/* The KV cache of 復刻 ChatGPT 有多難？ (jxzklqfsx.com), section
 * 為什么可以訓練如此之快 (the KV-cache paragraph: keys and values of earlier
 * positions are kept so decode does not recompute them) and of the CSDN nanochat
 * article (wap.jaobe.com), inference paragraph (the Engine's cache, filled by
 * prefill and extended by each decode step).
 * Creates a cache for `batch` sequences of up to t_max positions (t_max <= cfg
 * max_seq). mem == NULL: the library allocates and owns the memory. Otherwise
 * mem is a caller-owned device buffer of nc_kv_cache_bytes() bytes (256-byte
 * aligned) that must outlive the cache. Starts with length 0. */
NC_API nc_status nc_kv_cache_alloc(const nc_model* m, int32_t batch, int32_t t_max, void* mem,
                                   nc_kv_cache** out);
/* The same cache (jxzklqfsx.com, KV-cache paragraph) seen from outside: device
 * pointers to the K and V arrays, the number of filled positions, and the batch
 * and t_max it was created with. Any output pointer may be NULL. Returns
 * NC_ERR_INVALID_ARG for a NULL cache. */
NC_API nc_status nc_kv_cache_view(const nc_kv_cache* c, void** k, void** v, int32_t* len,
                                  int32_t* batch, int32_t* t_max);
NC_API void nc_kv_cache_free(nc_kv_cache* c);

/* Prefill: runs tokens (dev int32 [B, T]) from position 0 through the model,
 * writes K/V of positions 0..T-1 of sequences 0..B-1 into the cache and sets its
 * length to T. logits (dev fp32 [B, T, vocab]) receives every position's
 * logits. Requires 1 <= B <= cache batch, B <= max_batch, 1 <= T <= cache t_max.
 * (CSDN nanochat article, Engine paragraph: the prefill phase.) */
NC_API nc_status nc_prefill(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                            float* logits, nc_kv_cache* c, void* stream);

/* Continues a prefill: runs tokens (dev int32 [B, T]) at positions L..L+T-1,
 * where L is the cache's current length (the same for all its sequences), with
 * attention over positions 0..L+T-1 of the cache. Writes their K/V, sets the
 * length to L + T, and writes the T positions' logits (dev fp32 [B, T, vocab]).
 * L = 0 is nc_prefill; calling it in pieces gives the same K/V and logits as one
 * call over the whole sequence (up to the summation order of fp32 sums). T = 1 is
 * one decode step through the per-kernel path. Requires the bounds of nc_prefill
 * and L + T <= cache t_max; NC_ERR_UNSUPPORTED for T > 1 with L > 0 on an fp32
 * model. (CSDN nanochat article, Engine paragraph: prefill and decode over a
 * KV cache; the pages do not fix how a prompt is split.) */
NC_API nc_status nc_prefill_continue(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                                     float* logits, nc_kv_cache* c, void* stream);

/* As nc_prefill, but the LM head runs only on position T-1 of each sequence:
 * logits_last (dev fp32 [B, vocab], may be NULL) and argmax_out (dev int32 [B],
 * may be NULL; the greedy next token, lowest index on ties). */
NC_API nc_status nc_prefill_last(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                                 float* logits_last, int32_t* argmax_out, nc_kv_cache* c,
                                 void* stream);

/* Loss of a training step's forward pass (Microgpt summary, section 训练过程,
 * item 2: every position predicts the next token, and the loss is the
 * cross-entropy between that prediction and the true token). Runs the prefill of
 * nc_prefill over tokens (dev int32 [B, T]) and, per position r = b * T + t,
 *   loss[r] = log(sum_v exp(z[r, v])) - z[r, targets[r]],  z = that position's logits,
 * with the mean over the counted positions in *mean (dev fp32 [1]; NaN if none
 * counts). targets (dev int32 [B, T]): the true next token of each position; a
 * negative target leaves the position out (loss 0, not counted); a target >=
 * vocab does the same and sets NC_ERR_BOUNDS in the status word (nc_model_check).
 * loss (dev fp32 [B, T]) may be NULL. The logits are never stored: the LM-head
 * GEMM's epilogue reduces each row's 256-column blocks to (max, sum of exp) and
 * keeps the target's logit. The cache is written as by nc_prefill and is the
 * caller's. A model-owned scratch of B*T*(8*ceil(vocab/256) + 8) bytes is
 * allocated on the first call (and again for a larger B*T). The mean is summed in a
 * fixed order; the losses follow the projections' fp32 sums. Bounds as
 * nc_prefill; NC_ERR_INVALID_ARG for NULL targets or mean or pointers that are not
 * 4-byte aligned; NC_ERR_UNSUPPORTED for an fp32 model; NC_ERR_OOM if the scratch
 * cannot be allocated. */
NC_API nc_status nc_prefill_loss(nc_model* m, const int32_t* tokens, const int32_t* targets,
                                 int32_t B, int32_t T, float* loss, float* mean, nc_kv_cache* c,
                                 void* stream);

/* One decode step: token (dev int32 [B]) of each sequence at position pos, which
 * must equal the cache length; K/V are appended at pos, attention runs over
 * positions 0..pos, the cache length becomes pos+1. logits (dev fp32 [B, vocab],
 * may be NULL if argmax_out is given) and argmax_out (dev int32 [B] or NULL;
 * may alias tokens). (jxzklqfsx.com, KV cache paragraph; Microgpt summary 推理.) */
NC_API nc_status nc_decode_step(nc_model* m, const int32_t* tokens, int32_t B, int32_t pos,
                                float* logits, int32_t* argmax_out, nc_kv_cache* c, void* stream);

/* How nc_decode_step runs on the 16-bit path.
 *   NC_DECODE_AUTO        the persistent kernel where the shape allows it
 *                         (head_dim 128, n_head / n_kv_head <= 16, d_model and
 *                         d_mlp multiples of 128, vocab a multiple of 4), else
 *                         one kernel per projection / attention / norm.
 *   NC_DECODE_PERSISTENT  always the persistent kernel (NC_ERR_UNSUPPORTED where
 *                         the shape does not allow it).
 *   NC_DECODE_KERNELS     always one kernel per step of the block.
 * The persistent kernel runs a whole decode step for up to 32 sequences as one
 * cooperative launch with one CTA per SM: a producer warp streams every weight
 * matrix (packed once, on first use, into a model-owned copy of 16 KB units in
 * the tensor core's swizzled layout) and the KV cache through shared memory, two
 * MMA threads run the projections on tcgen05, and eight warps compute the
 * phases of the step between grid-wide barriers. Larger batches run as
 * several launches of up to 32 sequences. Projection partial sums are added in
 * fp32 in a run-dependent order. The fp32 path always uses kernels. */
typedef enum { NC_DECODE_AUTO = 0, NC_DECODE_PERSISTENT = 1, NC_DECODE_KERNELS = 2 } nc_decode_path;
NC_API nc_status nc_model_set_decode_path(nc_model* m, nc_decode_path path);

/* Greedy generation with HOST buffers: copies prompt (host int32 [B, T]) to the
 * device, prefills (token 0 = argmax of the last prompt position), then runs
 * `steps` decode steps, step j feeding token j back at position T + j and
 * producing token j + 1. Copies the steps + 1 generated tokens to out_tokens
 * (host int32 [steps + 1, B], step-major). The cache must hold T + steps
 * positions; it is overwritten from position 0. Synchronises `stream` before
 * returning. Host buffers may be pageable; pinned memory lets the copies run
 * asynchronously. */
NC_API nc_status nc_generate_host(nc_model* m, const int32_t* prompt, int32_t B, int32_t T,
                                  int32_t steps, int32_t* out_tokens, nc_kv_cache* c, void* stream);

/* Sets the cache length back to len (0 <= len <= current length): positions
 * >= len count as empty again and are overwritten by the next prefill / decode
 * steps (e.g. to roll back rejected tokens, or to replay a decode window). */
NC_API nc_status nc_kv_cache_set_length(nc_kv_cache* c, int32_t len);

/* Per-sequence cache lengths (the KV cache of jxzklqfsx.com, KV-cache paragraph,
 * kept for sequences of different lengths, as an Engine serving several requests
 * does: CSDN nanochat article, wap.jaobe.com, inference paragraph).
 * Every prefill / decode call sets the lengths of the sequences it ran; the
 * uniform calls (nc_prefill_continue, nc_decode_step) need all of their B
 * sequences at the same length. nc_kv_cache_set_lengths shortens sequences
 * [0, n) to lens[b] (host int32 [n]; each 0 <= lens[b] <= its current length;
 * NC_ERR_INVALID_ARG otherwise, nothing changed): a batch prefilled to a common
 * padded length T becomes ragged by cutting each sequence back to its own prompt
 * length (causal attention makes the kept rows independent of the cut ones).
 * nc_kv_cache_lengths copies the lengths of sequences [0, n) to lens (host). The
 * largest length is what nc_kv_cache_view reports. */
NC_API nc_status nc_kv_cache_set_lengths(nc_kv_cache* c, const int32_t* lens, int32_t n);
NC_API nc_status nc_kv_cache_lengths(const nc_kv_cache* c, int32_t* lens, int32_t n);

/* One decode step that also draws each sequence's next token (Microgpt summary,
 * section 推理（生成）, items 1-2: the next token is drawn from the predicted
 * distribution, the logits divided by a temperature first). As nc_decode_step
 * for tokens, B, pos and the cache, then next_out[b] (dev int32 [B], may alias
 * tokens) = the smallest index k whose cumulative probability under
 * softmax(logits[b] / temperature) exceeds u[b] (dev float [B], the caller's
 * uniforms in [0, 1); values outside are clamped) -- the inverse CDF, so a run is
 * reproducible from its inputs. temperature <= 0 gives the greedy index (lowest
 * on ties) and u may be NULL. The draw happens inside the step: every SM keeps
 * the logits of its whole vocabulary row groups in tensor memory, merges its
 * softmax partials with the others' and the SM whose share of the cumulative
 * distribution holds u scans its rows, so the logits are never written unless
 * `logits` (dev fp32 [B, V], may be NULL) asks for them. Sums are fp32: where u
 * lies within rounding of a cumulative boundary the neighbouring index may be
 * drawn. Persistent path only (NC_ERR_UNSUPPORTED otherwise, or for a
 * vocabulary above 6 * 128 rows per SM). */
NC_API nc_status nc_decode_step_sample(nc_model* m, const int32_t* tokens, int32_t B, int32_t pos,
                                       float temperature, const float* u, int32_t* next_out,
                                       float* logits, nc_kv_cache* c, void* stream);

/* nc_generate_host with sampling: prompt and out_tokens as there; u (HOST float
 * [steps + 1, B]) holds the uniforms, row 0 for the token after the prompt
 * (drawn from the prefill's last logits by the nc_op_sample kernel), row j + 1
 * for decode step j (nc_decode_step_sample). temperature <= 0: greedy, u may be
 * NULL. */
NC_API nc_status nc_generate_host_sample(nc_model* m, const int32_t* prompt, int32_t B, int32_t T,
                                         int32_t steps, float temperature, const float* u,
                                         int32_t* out_tokens, nc_kv_cache* c, void* stream);

/* One decode step with a position per sequence (jxzklqfsx.com, KV-cache
 * paragraph; CSDN nanochat article, Engine paragraph): sequence b's token
 * tokens[b] (dev int32 [B]) sits at position pos[b] (HOST int32 [B]), which must
 * equal that sequence's cache length; its K/V are written at pos[b], it attends
 * over positions 0..pos[b] with RoPE at pos[b], and its length becomes
 * pos[b] + 1. Outputs as nc_decode_step. Runs on the persistent kernel only:
 * NC_ERR_UNSUPPORTED for fp32 models, shapes the persistent kernel does not
 * take, or a model switched to NC_DECODE_KERNELS. NC_ERR_INVALID_ARG (nothing
 * enqueued) when a position differs from its cache length, is 0, or leaves no
 * room (pos[b] + 1 > t_max). */
NC_API nc_status nc_decode_step_ragged(nc_model* m, const int32_t* tokens, const int32_t* pos,
                                       int32_t B, float* logits, int32_t* argmax_out,
                                       nc_kv_cache* c, void* stream);

/* Synchronises `stream`, reads and clears the device status word. Returns NC_OK,
 * NC_ERR_DEVICE_TIMEOUT, NC_ERR_BOUNDS or NC_ERR_RANGE, in that order of
 * precedence (or NC_ERR_CUDA). */
NC_API nc_status nc_model_check(nc_model* m, void* stream);

/* ------------------------------------------------------------------------
 * Single-step entry points (the kernels of the path, one call each). Same
 * conventions; they allocate nothing unless stated.
 * ---------------------------------------------------------------------- */

/* y[m, :] = x[m, :] / sqrt(mean_j x[m, j]^2 + eps); x dev fp32 [M, d]; y dev
 * [M, d] in y_dtype (any of the three). d % 4 == 0. */
NC_API nc_status nc_op_rmsnorm(const float* x, void* y, nc_dtype y_dtype, int64_t M, int32_t d,
                               float eps, void* stream);

/* C = A B^T: A dev [M, K], B dev [N, K] in `dtype`, C dev fp32 [M, N]. bf16 and
 * f16 run the tcgen05 tensor-core GEMM (K % 64 == 0, N % 16 == 0); f32 runs the
 * CUDA-core GEMM. */
NC_API nc_status nc_op_gemm(const void* A, const void* B, float* C, int32_t M, int32_t N,
                            int32_t K, nc_dtype dtype, void* stream);

/* Causal attention over positions 0..T-1 of B sequences.
 * q dev [B, H, T, hd]; k, v dev [B, Hkv, t_max, hd] (positions 0..T-1 used);
 * o dev [B, T, H*hd]. Query head h reads KV head h / (H / Hkv). Scale 1/sqrt(hd). */
NC_API nc_status nc_op_attention_prefill(const void* q, const void* k, const void* v, void* o,
                                         int32_t B, int32_t H, int32_t Hkv, int32_t T,
                                         int32_t t_max, int32_t hd, nc_dtype dtype, void* stream);

/* Attention of one query per sequence (decode) over cache positions 0..len-1.
 * q dev [B, H, hd]; k, v dev [B, Hkv, t_max, hd]; o dev [B, H*hd]. Splits the
 * positions into ranges whose partial softmax states go to `scratch` (dev,
 * caller-owned, at least nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)
 * bytes, an upper bound for every len <= t_max) and are merged by log-sum-exp.
 * 16-bit types with hd 128 and H/Hkv <= 16 run on tensor cores (mma.sync; one
 * pass over K/V serves all query heads of a KV head); others on CUDA cores. */
NC_API size_t nc_op_attention_decode_scratch_bytes(int32_t B, int32_t H, int32_t t_max, int32_t hd);
NC_API nc_status nc_op_attention_decode(const void* q, const void* k, const void* v, void* o,
                                        int32_t B, int32_t H, int32_t Hkv, int32_t len,
                                        int32_t t_max, int32_t hd, nc_dtype dtype, void* scratch,
                                        size_t scratch_bytes, void* stream);

/* The same decode attention for callers that cannot allocate device memory
 * (an engine that owns all device memory through its own pool and forbids side
 * allocations, a plugin inside such a host, a latency-critical loop that cannot
 * take an allocation's implicit synchronisation). The paper has no counterpart:
 * this is a deployment variant. Arguments as nc_op_attention_decode, without the
 * scratch buffer: the split partial states go to one fixed 8 MiB array in the
 * library's device memory, held on every GPU that loads the library until the
 * process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - B * H * splits * (head_dim + 2) * 4 bytes must fit in 8 MiB (splits: the
 *     key range is cut so that about 2 CTAs per SM are busy, at most 64 and at
 *     most ceil(len / 64)); larger calls return NC_ERR_INVALID_ARG and
 *     nc_last_error() says how much was needed.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     Each call writes every partial state it reads, so nothing needs clearing,
 *     but calls that overlap on the GPU (other streams, other threads) race on
 *     the array: serialise them. */
NC_API nc_status nc_op_attention_decode_noalloc(const void* q, const void* k, const void* v,
                                                void* o, int32_t B, int32_t H, int32_t Hkv,
                                                int32_t len, int32_t t_max, int32_t hd,
                                                nc_dtype dtype, void* stream);

/* out[r] = index of the largest x[r, :] (lowest index on ties); x dev fp32
 * [rows, n], out dev int32 [rows]. */
NC_API nc_status nc_op_argmax(const float* x, int32_t rows, int32_t n, int32_t* out, void* stream);

/* Temperature sampling (Microgpt summary, section 推理（生成）, items 1 and 2: draw
 * the next token from the predicted distribution; the temperature divides the
 * logits, a lower one sharpening the distribution, a higher one flattening it).
 * out[r] = the smallest k with sum_{v <= k} p[r, v] > u[r], where
 * p[r, :] = softmax(logits[r, :] / temperature) (inverse CDF; fp32 arithmetic,
 * row max subtracted first; the last index if rounding leaves every partial sum at
 * or below u[r] Z). temperature <= 0 gives the greedy index (lowest on ties).
 * logits dev fp32 [rows, n]; u dev fp32 [rows]: the caller's random numbers, one
 * per row, clamped into [0, 1); out dev int32 [rows]. Nothing is allocated. Errors:
 * NC_ERR_INVALID_ARG for a NULL pointer, rows < 0 or n <= 0. */
NC_API nc_status nc_op_sample(const float* logits, int32_t rows, int32_t n, float temperature,
                              const float* u, int32_t* out, void* stream);

/* ------------------------------------------------------------------------
 * fp8 projection variant. The pages name fp8 only as a current topic of the
 * project (一天一个开源项目（第22篇）：nanochat, m.alixixi.com, section 项目简介, the
 * "版本" bullet) and define no format or scaling; the readings here: E4M3 without
 * infinities (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest
 * finite value 448), rounding to nearest with ties to the even mantissa,
 * saturating; a matrix is scaled per row by max|row| / 448 (1 for a zero row),
 * computed in fp32. The product runs on the tensor cores (tcgen05, kind::f8f6f4)
 * with fp32 accumulation: half the weight bytes of the 16-bit path.
 * ---------------------------------------------------------------------- */

/* scale[r] = max_c |x[r, c]| / 448 (1 if the row is zero) and q[r, c] =
 * E4M3(x[r, c] / scale[r]) (one byte each, nearest-even, saturating; the division
 * is IEEE fp32). x dev [rows, cols] in dtype (NC_F32, NC_BF16 or NC_F16); q dev
 * uint8 [rows, cols]; scale dev fp32 [rows]. cols % 16 == 0. Errors:
 * NC_ERR_INVALID_ARG for NULL or misaligned pointers or bad sizes. */
NC_API nc_status nc_op_quantize_e4m3(const void* x, nc_dtype dtype, int64_t rows, int32_t cols,
                                     uint8_t* q, float* scale, void* stream);

/* ------------------------------------------------------------------------
 * Next-token loss of a matrix product (the LM head of nc_prefill_loss as a
 * single step). Microgpt summary, section 训练过程, item 2.
 * ---------------------------------------------------------------------- */

/* Device scratch that nc_op_cross_entropy needs for M rows and N columns. */
NC_API size_t nc_op_cross_entropy_scratch_bytes(int32_t M, int32_t N);

/* loss[r] = log(sum_n exp(z[r, n])) - z[r, targets[r]] for z = A B^T (A dev
 * [M, K], B dev [N, K], both dtype NC_BF16 or NC_F16, row-major, fp32
 * accumulation on tcgen05), and *mean the mean over the rows counted. A row whose
 * target (dev int32 [M]) is outside [0, N) is left out (loss 0). The product is
 * reduced in the GEMM's epilogue per row and block of 256 columns; z is never
 * stored. loss dev fp32 [M] or NULL; mean dev fp32 [1] (NaN if no row counts);
 * scratch dev of at least nc_op_cross_entropy_scratch_bytes(M, N) bytes, owned by
 * the caller. K % 64 == 0 (N is free); A, B and scratch 16-byte aligned.
 * Errors: NC_ERR_INVALID_ARG for NULL or misaligned pointers, bad sizes or dtype,
 * or a small scratch; NC_ERR_UNSUPPORTED for K not a multiple of 64. */
NC_API nc_status nc_op_cross_entropy(const void* A, const void* B, const int32_t* targets,
                                     int32_t M, int32_t N, int32_t K, nc_dtype dtype, float* loss,
                                     float* mean, void* scratch, size_t scratch_bytes,
                                     void* stream);

/* Device scratch that nc_op_gemv_e4m3 needs for N features, K inputs, B tokens. */
NC_API size_t nc_op_gemv_e4m3_scratch_bytes(int32_t N, int32_t K, int32_t B);

/* y[t, n] = w_scale[n] * s_t * sum_k wq[n, k] * E4M3(x[t, k] / s_t), the
 * activations scaled per token as nc_op_quantize_e4m3 does: a decode step's
 * projection with fp8 weights (wq, w_scale from nc_op_quantize_e4m3 on W [N, K]).
 * wq dev [N, K] E4M3 codes, w_scale dev fp32 [N], x dev fp32 [B, K], y dev fp32
 * [B, N]; 1 <= B <= 128, K % 128 == 0, pointers 16-byte aligned; scratch dev of
 * at least nc_op_gemv_e4m3_scratch_bytes(N, K, B) bytes, owned by the caller
 * (not used by two calls at once). Nothing is allocated. Errors:
 * NC_ERR_INVALID_ARG for NULL or misaligned pointers, bad sizes or a small
 * scratch; NC_ERR_CUDA if a launch fails. */
NC_API nc_status nc_op_gemv_e4m3(const uint8_t* wq, const float* w_scale, int32_t N, int32_t K,
                                 const float* x, int32_t B, float* y, void* scratch,
                                 size_t scratch_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Measurement: per-kernel-class device time and a launch counter. Host-side
 * bookkeeping only; results are unchanged.
 * ---------------------------------------------------------------------- */
typedef enum {
    NC_K_EMBED = 0, NC_K_NORM, NC_K_QKV, NC_K_ATTN_PREFILL, NC_K_ATTN_DECODE, NC_K_OPROJ,
    NC_K_FC, NC_K_PROJ, NC_K_LM_HEAD, NC_K_ARGMAX, NC_K_DECODE_STEP, NC_K_COUNT
} nc_kernel_kind;

typedef struct {
    double ms;          /* summed device time (CUDA events on the launching stream) */
    int64_t launches;   /* kernel launches in this class */
} nc_kernel_time;

/* From now on the model records a CUDA event pair around each kernel class it
 * enqueues (one pair per projection / attention / norm call; a split-K
 * projection's finishing kernel counts with its GEMM). */
NC_API nc_status nc_profile_begin(nc_model* m);
/* Synchronises `stream`, sums the recorded intervals into out[NC_K_COUNT] and
 * stops recording. */
NC_API nc_status nc_profile_end(nc_model* m, void* stream, nc_kernel_time* out);
/* Number of kernels the library has launched in this process so far. */
NC_API int64_t nc_launch_count(void);

/* Phase timeline of the persistent decode step. While dev_buf (device uint64
 * [capacity], caller-owned) is set, every persistent step overwrites it with
 * %globaltimer readings (ns) taken by CTA 0: entry 0 at the start, entries
 * 2k-1 and 2k when it arrives at and leaves grid barrier k (k = 1 after the
 * embedding phase, then five per layer: after QKV, attention, O, FC, PROJ; then
 * after the final norm and after the LM head), and the last entry at the end.
 * Then, for the phase ending at barrier k, six marks at 2*nbar + 2 + 6(k-1) + m
 * (nbar = barriers per step): projections record m = 3 when they start staging
 * the activations, 0 when that is done, 1 when an accumulator has been read from
 * tensor memory and 2 after adding its partial sums (per row group; the last one
 * stays); attention records m = 0 after preparing q, 1 after the key tiles, 2
 * after adding its weighted softmax sums and 3 at the end, for each round of
 * (sequence, KV head) pairs it covers (later rounds overwrite earlier ones;
 * unused marks stay as they were); m = 4 is when CTA 0's producer started loading the phase's weights
 * or K/V tiles; m = 5 is unused. After those 8 * nbar + 2 entries, every CTA c < 256 of the launch
 * records, for barrier k, its arrival and exit time at 8 * nbar + 2 + 2 * (256 * (k - 1) + c)
 * (+ 1). capacity must be at least nc_decode_trace_entries(cfg), else nothing is
 * recorded. dev_buf NULL switches it off. Only the first 32 sequences' launch of
 * a step is traced. The readings cost one store each. */
NC_API nc_status nc_decode_trace(nc_model* m, uint64_t* dev_buf, int32_t capacity);
NC_API int32_t nc_decode_trace_entries(const nc_config* cfg);

#ifdef __cplusplus
}
#endif
#endif /* NC_H_ */
