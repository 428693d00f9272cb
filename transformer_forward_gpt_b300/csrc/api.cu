// C ABI of the library: argument checks, model / cache objects, workspace and
// the launch sequence of prefill and decode.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "decode_fused.h"
#include "nc_internal.h"
#include "tc.h"

namespace {

thread_local char g_err[512] = "";

void set_err(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

#define NC_CUDA(call)                                                              \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      set_err("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return NC_ERR_CUDA;                                                          \
    }                                                                              \
  } while (0)

#define NC_CHECK(cond, code, ...) \
  do {                            \
    if (!(cond)) {                \
      set_err(__VA_ARGS__);       \
      return code;                \
    }                             \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t dtype_size(nc_dtype d) { return d == NC_F32 ? 4 : 2; }
// number format of activations, Q and the KV cache
nc_dtype act_type(const nc_config& c) { return c.dtype == NC_F32 ? NC_F32 : c.act_dtype; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

nc_status check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_err("kernel launch failed: %s", cudaGetErrorString(e));
    return NC_ERR_CUDA;
  }
  return NC_OK;
}

std::atomic<int64_t> g_launches{0};

struct ProfRec {
  int kind;
  int64_t launches;
  cudaEvent_t a, b;
};

}  // namespace

namespace nc {
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
bool ensure_dyn_smem(const void* func, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> set_bytes;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = set_bytes[std::make_pair(func, dev)];
  if (have >= bytes) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  have = bytes;
  return true;
}
void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}
}  // namespace nc

struct nc_model {
  nc_config cfg;
  nc_dtype adt;              // activation / KV-cache format
  int device;
  const void* wte;
  const void* lm_head;
  std::vector<const void*> wq, wk, wv, wo, w_fc, w_proj;
  float* cos_tab = nullptr;  // [max_seq, hd/2]
  float* sin_tab = nullptr;
  float* cos_t = nullptr;    // [hd/2, max_seq]: consecutive positions adjacent
  float* sin_t = nullptr;
  uint32_t* status = nullptr;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float* x = nullptr;        // [Mmax, d] fp32 residual stream
  void* xn = nullptr;        // [Mmax, d] normalised activations
  void* q = nullptr;         // [Mmax, H*hd]
  void* att = nullptr;       // [Mmax, H*hd]
  void* h = nullptr;         // [Mmax, F]
  float* part = nullptr;     // split-K / fp32 projection outputs
  size_t part_elems = 0;
  float* xl = nullptr;       // [max_batch, d] last-position residual rows
  void* xnl = nullptr;       // [max_batch, d]
  float* logits_tmp = nullptr;  // [max_batch, V]
  int32_t* tok_dev = nullptr;   // [Mmax]
  int32_t* gen_dev = nullptr;   // [max_seq + 1, max_batch] generated tokens
  float* gen_u = nullptr;       // [max_seq + 1, max_batch] uniforms of a sampled generation
  float* attn_scratch = nullptr;
  size_t attn_scratch_bytes = 0;
  nc::TcModel* tc = nullptr;    // tensor-core state (16-bit models)
  void* wcopy = nullptr;        // weights converted to adt (when it differs from cfg.dtype)
  // persistent decode step (16-bit path), set up on first use
  int decode_path = NC_DECODE_AUTO;
  int sms = 0;
  nc::dec::Layout dlay{};
  uint8_t* dpack = nullptr;     // weights in 16 KB swizzled units
  void* dws = nullptr;          // its scratch
  float* d_qkv = nullptr;
  float* d_hacc = nullptr;
  float* d_ss = nullptr;
  void* d_xnf = nullptr;         // final-norm image of the LM head's B operand
  unsigned long long* d_amkey = nullptr;
  unsigned int* d_amcnt = nullptr;
  unsigned long long* d_bar = nullptr;
  float4* d_lm_part = nullptr;  // per-CTA softmax partials of the sampling mode
  float* d_att_num = nullptr;   // attention numerators [2][kMaxTok][H * head_dim]
  float* d_att_den = nullptr;   // and denominators [2][kMaxTok][H]
  // next-token loss (nc_prefill_loss), allocated on first use for the largest M
  void* ce_ws = nullptr;
  size_t ce_ws_bytes = 0;
  unsigned long long bar_base = 0;
  unsigned long long* dec_trace = nullptr;   // caller's buffer (nc_decode_trace)
  int32_t dec_trace_cap = 0;
  // measurement
  bool prof = false;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> event_pool;
};

namespace {
// Records a CUDA event pair around one kernel class while profiling is on.
struct ProfScope {
  nc_model* m;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  int64_t l0 = 0;
  cudaEvent_t take() {
    if (m->event_pool.empty()) {
      cudaEvent_t e;
      cudaEventCreate(&e);
      return e;
    }
    cudaEvent_t e = m->event_pool.back();
    m->event_pool.pop_back();
    return e;
  }
  ProfScope(nc_model* m_, int kind_, cudaStream_t s_) : m(m_), kind(kind_), s(s_) {
    if (!m->prof) return;
    a = take();
    cudaEventRecord(a, s);
    l0 = g_launches.load();
  }
  ~ProfScope() {
    if (!a) return;
    cudaEvent_t b = take();
    cudaEventRecord(b, s);
    m->recs.push_back({kind, g_launches.load() - l0, a, b});
  }
};
}  // namespace

struct nc_kv_cache {
  const nc_model* model;
  void* k = nullptr;
  void* v = nullptr;
  void* mem = nullptr;
  bool owns = false;
  int32_t batch = 0, t_max = 0, len = 0;   // len: the largest of lens
  std::vector<int32_t> lens;                 // filled positions of each sequence
  size_t layer_elems = 0;  // batch * Hkv * t_max * hd
  bool maps = false;       // TMA views of K and V for the persistent decode step
  CUtensorMap tmk, tmv;
};

extern "C" {

const char* nc_version(void) { return "nc-b300 0.1 (sm_103a)"; }

const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "ok";
    case NC_ERR_INVALID_ARG: return "invalid argument";
    case NC_ERR_UNSUPPORTED: return "unsupported shape";
    case NC_ERR_OOM: return "out of device memory";
    case NC_ERR_CUDA: return "CUDA error";
    case NC_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case NC_ERR_BOUNDS: return "token id out of range";
    case NC_ERR_RANGE: return "value out of fp16 range";
  }
  return "unknown status";
}

const char* nc_last_error(void) { return g_err; }

int64_t nc_param_count(const nc_config* c) {
  if (!c) return -1;
  const int64_t d = c->d_model, qd = (int64_t)c->n_head * c->head_dim,
                kvd = (int64_t)c->n_kv_head * c->head_dim, F = c->d_mlp;
  const int64_t per_layer = qd * d + 2 * kvd * d + d * qd + F * d + d * F;
  return 2 * (int64_t)c->vocab * d + (int64_t)c->n_layer * per_layer;
}

static nc_status validate_config(const nc_config* c) {
  NC_CHECK(c, NC_ERR_INVALID_ARG, "config is NULL");
  NC_CHECK(c->vocab > 0 && c->d_model > 0 && c->n_layer > 0 && c->n_head > 0 &&
               c->n_kv_head > 0 && c->head_dim > 0 && c->d_mlp > 0 && c->max_seq > 0 &&
               c->max_batch > 0,
           NC_ERR_INVALID_ARG, "config sizes must be positive");
  NC_CHECK(c->n_head % c->n_kv_head == 0, NC_ERR_INVALID_ARG,
           "n_head (%d) must be a multiple of n_kv_head (%d)", c->n_head, c->n_kv_head);
  NC_CHECK(c->head_dim % 2 == 0 && c->head_dim <= 128, NC_ERR_UNSUPPORTED,
           "head_dim must be even and <= 128");
  NC_CHECK(c->d_model % 4 == 0 && c->d_mlp % 4 == 0, NC_ERR_UNSUPPORTED,
           "d_model and d_mlp must be multiples of 4");
  NC_CHECK(c->rms_eps >= 0.f && c->rope_base > 0.f, NC_ERR_INVALID_ARG, "bad eps / rope base");
  NC_CHECK(c->dtype == NC_F32 || c->dtype == NC_BF16 || c->dtype == NC_F16, NC_ERR_INVALID_ARG,
           "bad dtype");
  if (c->dtype != NC_F32) {
    NC_CHECK(c->act_dtype == NC_BF16 || c->act_dtype == NC_F16, NC_ERR_INVALID_ARG,
             "act_dtype must be NC_BF16 or NC_F16 for 16-bit weights");
    NC_CHECK(c->head_dim == 128 && c->d_model % 64 == 0 && c->d_mlp % 64 == 0, NC_ERR_UNSUPPORTED,
             "tensor-core path needs head_dim 128 and d_model, d_mlp multiples of 64");
  }
  return NC_OK;
}

void nc_model_destroy(nc_model* m) {
  if (!m) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(m->device);
  if (m->tc) nc::tc_destroy(m->tc);
  for (auto& r : m->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : m->event_pool) cudaEventDestroy(e);
  cudaFree(m->wcopy);
  cudaFree(m->dpack);
  cudaFree(m->ce_ws);
  cudaFree(m->dws);
  cudaFree(m->ws);
  cudaFree(m->cos_tab);
  cudaFree(m->sin_tab);
  cudaFree(m->cos_t);
  cudaFree(m->sin_t);
  cudaFree(m->status);
  cudaSetDevice(prev);
  delete m;
}

nc_status nc_model_create(const nc_config* cfg, const nc_weights* w, nc_model** out) {
  NC_CHECK(out, NC_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  nc_status st = validate_config(cfg);
  if (st != NC_OK) return st;
  NC_CHECK(w && w->wte && w->lm_head && w->wq && w->wk && w->wv && w->wo && w->w_fc && w->w_proj,
           NC_ERR_INVALID_ARG, "weights struct has NULL members");
  const int L = cfg->n_layer;
  NC_CHECK(aligned16(w->wte) && aligned16(w->lm_head), NC_ERR_INVALID_ARG,
           "wte / lm_head must be 16-byte aligned");
  for (int l = 0; l < L; ++l) {
    const void* ps[6] = {w->wq[l], w->wk[l], w->wv[l], w->wo[l], w->w_fc[l], w->w_proj[l]};
    for (const void* p : ps)
      NC_CHECK(p && aligned16(p), NC_ERR_INVALID_ARG, "layer %d weight NULL or misaligned", l);
  }
  nc_model* m = new nc_model();
  m->cfg = *cfg;
  m->adt = act_type(*cfg);
  m->cfg.act_dtype = m->adt;
  cudaGetDevice(&m->device);
  m->wte = w->wte;
  m->lm_head = w->lm_head;
  m->wq.assign(w->wq, w->wq + L);
  m->wk.assign(w->wk, w->wk + L);
  m->wv.assign(w->wv, w->wv + L);
  m->wo.assign(w->wo, w->wo + L);
  m->w_fc.assign(w->w_fc, w->w_fc + L);
  m->w_proj.assign(w->w_proj, w->w_proj + L);

  auto fail = [&](nc_status s) {
    nc_model_destroy(m);
    return s;
  };
  // cos/sin tables: fp64 on the host, stored fp32 ("precomputed and kept in GPU memory")
  const int half = cfg->head_dim / 2, S = cfg->max_seq;
  // The position-minor copies serve the prefill Q/K epilogue, where the 32 lanes
  // of a warp hold 32 consecutive positions: one table entry for all of them is
  // one 128-byte line instead of 32.
  std::vector<float> c(size_t(S) * half), s(size_t(S) * half), ct(c.size()), snt(s.size());
  for (int t = 0; t < S; ++t)
    for (int i = 0; i < half; ++i) {
      const double theta = (double)t * pow((double)cfg->rope_base, -2.0 * i / cfg->head_dim);
      c[size_t(t) * half + i] = ct[size_t(i) * S + t] = (float)cos(theta);
      s[size_t(t) * half + i] = snt[size_t(i) * S + t] = (float)sin(theta);
    }
  if (cudaMalloc(&m->cos_tab, c.size() * 4) != cudaSuccess ||
      cudaMalloc(&m->sin_tab, s.size() * 4) != cudaSuccess ||
      cudaMalloc(&m->cos_t, ct.size() * 4) != cudaSuccess ||
      cudaMalloc(&m->sin_t, snt.size() * 4) != cudaSuccess ||
      cudaMalloc(&m->status, 256) != cudaSuccess) {
    set_err("allocation of tables failed");
    return fail(NC_ERR_OOM);
  }
  if (cudaMemcpy(m->cos_tab, c.data(), c.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(m->sin_tab, s.data(), s.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(m->cos_t, ct.data(), ct.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(m->sin_t, snt.data(), snt.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(m->status, 0, 256) != cudaSuccess) {
    set_err("upload of tables failed");
    return fail(NC_ERR_CUDA);
  }

  // workspace
  const size_t es = dtype_size(m->adt);
  const size_t Mmax = (size_t)cfg->max_batch * cfg->max_seq;
  const size_t d = cfg->d_model, qd = (size_t)cfg->n_head * cfg->head_dim, F = cfg->d_mlp;
  const size_t nqkv = (size_t)(cfg->n_head + 2 * cfg->n_kv_head) * cfg->head_dim;
  const size_t widest = std::max(std::max(nqkv, F), d);
  // fp32 path keeps every projection output in `part`; the bf16 path uses it
  // for split-K partials of the batch rows only.
  size_t part_elems = m->adt == NC_F32 ? Mmax * widest
                                           : (size_t)nc::kMaxSplits * nc::kSwapMaxRows * widest;
  m->part_elems = part_elems;
  m->attn_scratch_bytes =
      nc_op_attention_decode_scratch_bytes(cfg->max_batch, cfg->n_head, cfg->max_seq,
                                           cfg->head_dim);
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  const size_t o_x = carve(Mmax * d * 4), o_xn = carve(Mmax * d * es),
               o_q = carve(Mmax * qd * es), o_att = carve(Mmax * qd * es),
               o_h = carve(Mmax * F * es), o_part = carve(part_elems * 4),
               o_xl = carve((size_t)cfg->max_batch * d * 4),
               o_xnl = carve((size_t)cfg->max_batch * d * es),
               o_lt = carve((size_t)cfg->max_batch * cfg->vocab * 4), o_tok = carve(Mmax * 4),
               o_gen = carve(((size_t)cfg->max_seq + 1) * cfg->max_batch * 4),
               o_genu = carve(((size_t)cfg->max_seq + 1) * cfg->max_batch * 4),
               o_as = carve(m->attn_scratch_bytes);
  m->ws_bytes = off;
  if (cudaMalloc(&m->ws, m->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    set_err("workspace allocation of %zu bytes failed", m->ws_bytes);
    return fail(NC_ERR_OOM);
  }
  char* base = static_cast<char*>(m->ws);
  m->x = reinterpret_cast<float*>(base + o_x);
  m->xn = base + o_xn;
  m->q = base + o_q;
  m->att = base + o_att;
  m->h = base + o_h;
  m->part = reinterpret_cast<float*>(base + o_part);
  m->xl = reinterpret_cast<float*>(base + o_xl);
  m->xnl = base + o_xnl;
  m->logits_tmp = reinterpret_cast<float*>(base + o_lt);
  m->tok_dev = reinterpret_cast<int32_t*>(base + o_tok);
  m->gen_dev = reinterpret_cast<int32_t*>(base + o_gen);
  m->gen_u = reinterpret_cast<float*>(base + o_genu);
  m->attn_scratch = reinterpret_cast<float*>(base + o_as);

  if (m->adt != NC_F32) {
    if (m->adt != cfg->dtype) {
      // working copies of the projection / LM-head weights in the activation format
      const size_t kvd = (size_t)cfg->n_kv_head * cfg->head_dim;
      const size_t sizes[6] = {qd * d, kvd * d, kvd * d, d * qd, F * d, d * F};
      size_t bytes = round_up((size_t)cfg->vocab * d * 2, 256);
      for (int l = 0; l < L; ++l)
        for (size_t z : sizes) bytes += round_up(z * 2, 256);
      if (cudaMalloc(&m->wcopy, bytes) != cudaSuccess) {
        m->wcopy = nullptr;
        cudaGetLastError();
        set_err("weight copy allocation of %zu bytes failed", bytes);
        return fail(NC_ERR_OOM);
      }
      char* wp = static_cast<char*>(m->wcopy);
      auto conv = [&](const void*& ptr, size_t n) {
        nc::launch_convert16(ptr, cfg->dtype, wp, m->adt, (int64_t)n, 0);
        ptr = wp;
        wp += round_up(n * 2, 256);
      };
      for (int l = 0; l < L; ++l) {
        conv(m->wq[l], sizes[0]);
        conv(m->wk[l], sizes[1]);
        conv(m->wv[l], sizes[2]);
        conv(m->wo[l], sizes[3]);
        conv(m->w_fc[l], sizes[4]);
        conv(m->w_proj[l], sizes[5]);
      }
      conv(m->lm_head, (size_t)cfg->vocab * d);
      if (cudaDeviceSynchronize() != cudaSuccess) {
        set_err("weight conversion failed");
        return fail(NC_ERR_CUDA);
      }
    }
    st = nc::tc_create(m->cfg, m->lm_head, m->wq.data(), m->wk.data(), m->wv.data(), m->wo.data(),
                       m->w_fc.data(), m->w_proj.data(), m->xn, m->att, m->h, m->xnl, Mmax,
                       m->status, &m->tc);
    if (st != NC_OK) return fail(st);
  }
  *out = m;
  return NC_OK;
}

size_t nc_kv_cache_bytes(const nc_config* cfg, int32_t batch, int32_t t_max) {
  if (!cfg || batch <= 0 || t_max <= 0) return 0;
  const size_t per = (size_t)cfg->n_layer * batch * cfg->n_kv_head * t_max * cfg->head_dim *
                     dtype_size(act_type(*cfg));
  return 256 + 2 * round_up(per, 256);
}

nc_status nc_kv_cache_alloc(const nc_model* m, int32_t batch, int32_t t_max, void* mem,
                            nc_kv_cache** out) {
  NC_CHECK(m && out, NC_ERR_INVALID_ARG, "NULL model or out");
  *out = nullptr;
  NC_CHECK(batch > 0 && t_max > 0, NC_ERR_INVALID_ARG, "batch and t_max must be positive");
  NC_CHECK(t_max <= m->cfg.max_seq, NC_ERR_INVALID_ARG, "t_max %d exceeds max_seq %d", t_max,
           m->cfg.max_seq);
  NC_CHECK(!mem || (reinterpret_cast<uintptr_t>(mem) & 255u) == 0, NC_ERR_INVALID_ARG,
           "cache memory must be 256-byte aligned");
  const size_t bytes = nc_kv_cache_bytes(&m->cfg, batch, t_max);
  nc_kv_cache* c = new nc_kv_cache();
  c->model = m;
  c->batch = batch;
  c->t_max = t_max;
  c->layer_elems = (size_t)batch * m->cfg.n_kv_head * t_max * m->cfg.head_dim;
  c->lens.assign(batch, 0);
  if (!mem) {
    if (cudaMalloc(&c->mem, bytes) != cudaSuccess) {
      cudaGetLastError();
      delete c;
      set_err("KV cache allocation of %zu bytes failed", bytes);
      return NC_ERR_OOM;
    }
    c->owns = true;
  } else {
    c->mem = mem;
  }
  const size_t per = round_up((size_t)m->cfg.n_layer * c->layer_elems * dtype_size(m->adt), 256);
  c->k = static_cast<char*>(c->mem) + 256;
  c->v = static_cast<char*>(c->mem) + 256 + per;
  *out = c;
  return NC_OK;
}

nc_status nc_kv_cache_view(const nc_kv_cache* c, void** k, void** v, int32_t* len, int32_t* batch,
                           int32_t* t_max) {
  NC_CHECK(c, NC_ERR_INVALID_ARG, "cache is NULL");
  if (k) *k = c->k;
  if (v) *v = c->v;
  if (len) *len = c->len;
  if (batch) *batch = c->batch;
  if (t_max) *t_max = c->t_max;
  return NC_OK;
}

void nc_kv_cache_free(nc_kv_cache* c) {
  if (!c) return;
  if (c->owns) cudaFree(c->mem);
  delete c;
}

}  // extern "C"

// --------------------------------------------------------------- launch plan
namespace {

using nc::RowMap;
using nc::QkvDst;

void* layer_ptr(void* base, size_t layer_elems, int l, nc_dtype dt) {
  return static_cast<char*>(base) + (size_t)l * layer_elems * dtype_size(dt);
}

// Runs the transformer blocks over rows [M] (B sequences of `rows_per_seq`
// rows each, starting at position pos0). On entry m->x holds the embeddings and
// m->xn their RMSNorm; on exit m->x holds the final residual and m->xn its final
// RMSNorm.
nc_status run_blocks(nc_model* m, nc_kv_cache* c, int B, int rows_per_seq, int pos0,
                     cudaStream_t s) {
  const nc_config& cfg = m->cfg;
  const nc_dtype dt = m->adt;
  const int64_t M = (int64_t)B * rows_per_seq;
  const int H = cfg.n_head, Hkv = cfg.n_kv_head, hd = cfg.head_dim, d = cfg.d_model,
            F = cfg.d_mlp;
  const int nqkv = (H + 2 * Hkv) * hd;
  const bool decode = rows_per_seq == 1 && pos0 > 0;
  const bool tc = dt != NC_F32;
  RowMap rm{rows_per_seq, pos0};
  for (int l = 0; l < cfg.n_layer; ++l) {
    QkvDst dst{m->q, layer_ptr(c->k, c->layer_elems, l, dt), layer_ptr(c->v, c->layer_elems, l, dt),
               H, Hkv, hd, c->t_max, m->cos_tab, m->sin_tab, cfg.rms_eps,
               m->cos_t, m->sin_t, cfg.max_seq, m->status};
    // Q/K/V projections + RoPE + QK norm + cache write
    {
    ProfScope ps(m, NC_K_QKV, s);
    if (tc) {
      nc_status st = nc::tc_qkv(m->tc, l, M, rm, dst, m->part, s);
      if (st != NC_OK) return st;
    } else {
      const size_t kvd = (size_t)Hkv * hd;
      nc::launch_gemm_simt(m->xn, m->wq[l], m->part, M, H * hd, d, nqkv, dt, s);
      nc::launch_gemm_simt(m->xn, m->wk[l], m->part + (size_t)H * hd, M, Hkv * hd, d, nqkv, dt, s);
      nc::launch_gemm_simt(m->xn, m->wv[l], m->part + (size_t)H * hd + kvd, M, Hkv * hd, d, nqkv,
                           dt, s);
      nc::launch_qkv_post(m->part, 1, M, rm, dst, dt, s);
    }
    }
    // causal attention
    {
    ProfScope ps(m, decode ? NC_K_ATTN_DECODE : NC_K_ATTN_PREFILL, s);
    if (decode) {
      nc::launch_attention_decode(m->q, dst.k_cache, dst.v_cache, m->att, B, H, Hkv, pos0 + 1,
                                  c->t_max, hd, dt, m->attn_scratch, s);
    } else if (tc) {
      const int64_t one_layer = (int64_t)c->batch * Hkv * c->t_max * hd;
      nc_status st = nc::tc_attention_prefill_tc(m->q, dst.k_cache, dst.v_cache, m->att, B, H,
                                                 Hkv, rows_per_seq, pos0, c->t_max, 1, one_layer,
                                                 0, dt, m->status, s);
      // descriptors could not be built: the mma.sync kernel needs none (it serves
      // prefill from position 0 only)
      if (st != NC_OK && pos0 == 0)
        st = nc::tc_attention_prefill(m->q, dst.k_cache, dst.v_cache, m->att, B, H, Hkv,
                                      rows_per_seq, c->t_max, dt, s);
      if (st != NC_OK) return st;
    } else {
      nc::launch_attention_prefill_simt(m->q, dst.k_cache, dst.v_cache, m->att, B, H, Hkv,
                                        rows_per_seq, c->t_max, hd, dt, s);
    }
    }
    // output projection + residual, then the pre-MLP RMSNorm
    if (tc) {
      nc_status st;
      {
        ProfScope ps(m, NC_K_OPROJ, s);
        st = nc::tc_out_proj(m->tc, l, M, m->x, m->part, s);
      }
      if (st != NC_OK) return st;
      {
        ProfScope ps(m, NC_K_NORM, s);
        nc::launch_rmsnorm(m->x, m->xn, dt, M, d, cfg.rms_eps, s);
      }
      {
        ProfScope ps(m, NC_K_FC, s);
        st = nc::tc_fc(m->tc, l, M, m->part, s);
      }
      if (st != NC_OK) return st;
      {
        ProfScope ps(m, NC_K_PROJ, s);
        st = nc::tc_proj(m->tc, l, M, m->x, m->part, s);
      }
      if (st != NC_OK) return st;
      {
        ProfScope ps(m, NC_K_NORM, s);
        nc::launch_rmsnorm(m->x, m->xn, dt, M, d, cfg.rms_eps, s);
      }
    } else {
      nc::launch_gemm_simt(m->att, m->wo[l], m->part, M, d, H * hd, d, dt, s);
      nc::launch_residual_finish(m->part, 1, m->x, M, d, m->xn, dt, cfg.rms_eps, s);
      nc::launch_gemm_simt(m->xn, m->w_fc[l], m->part, M, F, d, F, dt, s);
      nc::launch_relu2_finish(m->part, 1, m->h, M, F, dt, m->status, s);
      nc::launch_gemm_simt(m->h, m->w_proj[l], m->part, M, d, F, d, dt, s);
      nc::launch_residual_finish(m->part, 1, m->x, M, d, m->xn, dt, cfg.rms_eps, s);
    }
  }
  return check_launch();
}

// logits[M, V] = xn[M, d] lm_head^T
nc_status run_lm_head(nc_model* m, const void* xn, int64_t M, float* logits, cudaStream_t s) {
  ProfScope ps(m, NC_K_LM_HEAD, s);
  if (m->adt != NC_F32) return nc::tc_lm_head(m->tc, xn, M, logits, m->part, s);
  nc::launch_gemm_simt(xn, m->lm_head, logits, M, m->cfg.vocab, m->cfg.d_model, m->cfg.vocab,
                       NC_F32, s);
  return check_launch();
}

nc_status check_prefill_args(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                             nc_kv_cache* c) {
  NC_CHECK(m && c && tokens, NC_ERR_INVALID_ARG, "NULL model, cache or tokens");
  NC_CHECK(c->model == m, NC_ERR_INVALID_ARG, "cache belongs to another model");
  NC_CHECK(B >= 1 && B <= c->batch && B <= m->cfg.max_batch, NC_ERR_INVALID_ARG,
           "B=%d out of range (cache batch %d, max_batch %d)", B, c->batch, m->cfg.max_batch);
  NC_CHECK(T >= 1 && T <= c->t_max && T <= m->cfg.max_seq, NC_ERR_INVALID_ARG,
           "T=%d out of range (cache t_max %d)", T, c->t_max);
  NC_CHECK(aligned16(tokens) || (reinterpret_cast<uintptr_t>(tokens) & 3u) == 0,
           NC_ERR_INVALID_ARG, "tokens must be 4-byte aligned");
  return NC_OK;
}

// Sets the lengths of sequences [0, B) to n and len to the largest length.
void set_lens(nc_kv_cache* c, int32_t B, int32_t n) {
  for (int32_t b = 0; b < B; ++b) c->lens[b] = n;
  c->len = *std::max_element(c->lens.begin(), c->lens.end());
}
// True when sequences [0, B) all hold n positions.
bool lens_equal(const nc_kv_cache* c, int32_t B, int32_t n) {
  for (int32_t b = 0; b < B; ++b)
    if (c->lens[b] != n) return false;
  return true;
}

// Runs T positions of B sequences starting at absolute position pos0 (the cache
// already holds positions 0..pos0-1) and sets their cache lengths to pos0 + T.
nc_status prefill_common(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                         nc_kv_cache* c, cudaStream_t s, int32_t pos0 = 0) {
  const int64_t M = (int64_t)B * T;
  {
    ProfScope ps(m, NC_K_EMBED, s);
    nc::launch_embed_norm(tokens, m->wte, m->cfg.dtype, m->x, m->xn, m->adt, M, m->cfg.d_model,
                          m->cfg.vocab, m->cfg.rms_eps, m->status, s);
  }
  nc_status st = run_blocks(m, c, B, T, pos0, s);
  if (st != NC_OK) return st;
  set_lens(c, B, pos0 + T);
  return NC_OK;
}


// ------------------------------------------------ persistent decode step
bool decode_fused_applies(const nc_model* m) {
  const nc_config& c = m->cfg;
  if (m->adt == NC_F32 || c.vocab % 4 != 0) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return false;
  return nc::dec::supported(c.d_model, c.n_head, c.n_kv_head, c.d_mlp, c.head_dim, c.vocab, sms);
}

nc_status decode_fused_init(nc_model* m, cudaStream_t s) {
  if (m->dpack) return NC_OK;
  const nc_config& c = m->cfg;
  int dev = 0;
  NC_CUDA(cudaGetDevice(&dev));
  NC_CUDA(cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, dev));
  int coop = 0;
  NC_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
  NC_CHECK(coop, NC_ERR_UNSUPPORTED, "device has no cooperative launch");
  m->dlay = nc::dec::layout_of(c.n_layer, c.d_model, c.n_head, c.n_kv_head, c.d_mlp, c.vocab);
  const int K = nc::dec::kMaxTok;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t o_qkv = carve((size_t)2 * K * m->dlay.nqkv_pad * 4),
               o_h = carve((size_t)K * c.d_mlp * 4), o_ss = carve((size_t)2 * c.n_layer * K * 4),
               o_xnf = carve((size_t)m->dlay.xn_img_bytes),
               o_key = carve((size_t)K * 8), o_amc = carve((size_t)K * 4), o_bar = carve(8),
               o_lmp = carve((size_t)nc::dec::kMaxAttnBlocks * K * 16),
               o_an = carve((size_t)2 * K * c.n_head * c.head_dim * 4),
               o_ad = carve((size_t)2 * K * c.n_head * 4);
  if (cudaMalloc(&m->dws, off) != cudaSuccess) {
    cudaGetLastError();
    m->dws = nullptr;
    set_err("decode scratch allocation of %zu bytes failed", off);
    return NC_ERR_OOM;
  }
  NC_CUDA(cudaMemset(m->dws, 0, off));
  char* b = static_cast<char*>(m->dws);
  m->d_qkv = reinterpret_cast<float*>(b + o_qkv);
  m->d_hacc = reinterpret_cast<float*>(b + o_h);
  m->d_ss = reinterpret_cast<float*>(b + o_ss);
  m->d_xnf = b + o_xnf;
  m->d_amkey = reinterpret_cast<unsigned long long*>(b + o_key);
  m->d_amcnt = reinterpret_cast<unsigned int*>(b + o_amc);
  m->d_bar = reinterpret_cast<unsigned long long*>(b + o_bar);
  m->d_lm_part = reinterpret_cast<float4*>(b + o_lmp);
  m->d_att_num = reinterpret_cast<float*>(b + o_an);
  m->d_att_den = reinterpret_cast<float*>(b + o_ad);
  m->bar_base = 0;
  uint8_t* pack = nullptr;
  if (cudaMalloc(&pack, (size_t)m->dlay.total_bytes) != cudaSuccess) {
    cudaGetLastError();
    set_err("packed decode weights: allocation of %lld bytes failed",
            (long long)m->dlay.total_bytes);
    return NC_ERR_OOM;
  }
  nc::dec::PackSrc src{c.n_layer, c.d_model, c.n_head, c.n_kv_head, c.d_mlp, c.vocab,
                       m->wq.data(), m->wk.data(), m->wv.data(), m->wo.data(),
                       m->w_fc.data(), m->w_proj.data(), m->lm_head};
  nc_status st = nc::dec::pack_weights(src, m->adt == NC_F16, pack, s);
  if (st != NC_OK) {
    cudaFree(pack);
    set_err("packing the decode weights failed");
    return st;
  }
  m->dpack = pack;
  return NC_OK;
}

// Sampling of the persistent step: off (greedy index from the logits in memory),
// or drawn inside the step from whole vocabulary row groups kept on chip.
struct StepSample {
  bool on = false;
  float temperature = 0.f;   // <= 0: greedy index
  const float* u = nullptr;  // dev [B]
};

// One persistent decode step for B sequences; sequence b's new token sits at
// position pos[b] (host array), which is also its cache length.
nc_status decode_fused(nc_model* m, const int32_t* tokens, int32_t B, const int32_t* pos,
                       float* logits, int32_t* argmax_out, nc_kv_cache* c, cudaStream_t s,
                       const StepSample& smp = StepSample()) {
  nc_status st = decode_fused_init(m, s);
  if (st != NC_OK) return st;
  const nc_config& cfg = m->cfg;
  const bool f16 = m->adt == NC_F16;
  if (!c->maps) {
    const uint64_t rows = (uint64_t)cfg.n_layer * c->batch * cfg.n_kv_head * c->t_max;
    NC_CHECK(nc::dec::make_cache_map(&c->tmk, c->k, rows, f16) &&
                 nc::dec::make_cache_map(&c->tmv, c->v, rows, f16),
             NC_ERR_CUDA, "TMA descriptors of the KV cache could not be built");
    c->maps = true;
  }
  ProfScope ps(m, NC_K_DECODE_STEP, s);
  for (int b0 = 0; b0 < B; b0 += nc::dec::kMaxTok) {
    const int Bc = std::min(nc::dec::kMaxTok, B - b0);
    nc::dec::Params p{};
    p.B = Bc;
    p.b_off = b0;
    for (int i = 0; i < Bc; ++i) p.pos[i] = pos[b0 + i];
    p.cache_batch = c->batch;
    p.t_max = c->t_max;
    p.L = cfg.n_layer;
    p.d = cfg.d_model;
    p.H = cfg.n_head;
    p.Hkv = cfg.n_kv_head;
    p.F = cfg.d_mlp;
    p.V = cfg.vocab;
    p.vpad = m->dlay.vpad;
    p.nqkv = m->dlay.nqkv;
    p.nqkv_pad = m->dlay.nqkv_pad;
    NC_CHECK(nc::dec::plan_attention(p, m->sms) > 0, NC_ERR_UNSUPPORTED,
             "decode attention work too large");
    p.eps = cfg.rms_eps;
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)cfg.head_dim));
    p.layer_bytes = m->dlay.layer_bytes;
    p.off_o = m->dlay.off_o;
    p.off_fc = m->dlay.off_fc;
    p.off_proj = m->dlay.off_proj;
    p.tokens = tokens + b0;
    p.argmax_out = argmax_out ? argmax_out + b0 : nullptr;
    p.wte = m->wte;
    p.wpack = m->dpack;
    p.cos_tab = m->cos_tab;
    p.sin_tab = m->sin_tab;
    p.k_cache = c->k;
    p.v_cache = c->v;
    p.x = m->x;
    p.qkv_acc = m->d_qkv;
    p.hacc = m->d_hacc;
    p.ss = m->d_ss;
    p.xn_img = m->d_xnf;
    p.logits = (logits ? logits : m->logits_tmp) + (size_t)b0 * cfg.vocab;
    p.sample = smp.on ? 1 : 0;
    if (smp.on) {
      p.logits = logits ? logits + (size_t)b0 * cfg.vocab : nullptr;   // never written if NULL
      p.temp_k = smp.temperature > 0.f ? (float)(1.4426950408889634 / smp.temperature) : 0.f;
      p.u = smp.u ? smp.u + b0 : nullptr;
      p.lm_part = m->d_lm_part;
    }
    p.argmax_key = m->d_amkey;
    p.argmax_count = m->d_amcnt;
    p.bar_counter = m->d_bar;
    p.bar_base = m->bar_base;
    p.status = m->status;
    p.abort = m->status + 1;
    p.nbar = nc::dec::barriers_per_step(cfg.n_layer);
    p.trace = (b0 == 0 && m->dec_trace && m->dec_trace_cap >= nc::dec::trace_entries(cfg.n_layer))
                  ? m->dec_trace
                  : nullptr;
    p.att_num = m->d_att_num;
    p.att_den = m->d_att_den;
    st = nc::dec::launch_step(c->tmk, c->tmv, p, f16, cfg.dtype, m->sms, s);
    if (st != NC_OK) return st;
    m->bar_base += (unsigned long long)nc::dec::barriers_per_step(cfg.n_layer) * m->sms;
  }
  return NC_OK;
}
}  // namespace

extern "C" {

nc_status nc_prefill(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, float* logits,
                     nc_kv_cache* c, void* stream) {
  nc_status st = check_prefill_args(m, tokens, B, T, c);
  if (st != NC_OK) return st;
  NC_CHECK(logits && aligned16(logits), NC_ERR_INVALID_ARG, "logits NULL or misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = prefill_common(m, tokens, B, T, c, s);
  if (st != NC_OK) return st;
  return run_lm_head(m, m->xn, (int64_t)B * T, logits, s);
}

nc_status nc_prefill_continue(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                              float* logits, nc_kv_cache* c, void* stream) {
  nc_status st = check_prefill_args(m, tokens, B, T, c);
  if (st != NC_OK) return st;
  NC_CHECK(logits && aligned16(logits), NC_ERR_INVALID_ARG, "logits NULL or misaligned");
  const int32_t pos0 = c->lens[0];
  NC_CHECK(lens_equal(c, B, pos0), NC_ERR_INVALID_ARG,
           "continuing a prefill needs the same cache length for all %d sequences", B);
  NC_CHECK((int64_t)pos0 + T <= c->t_max && (int64_t)pos0 + T <= m->cfg.max_seq,
           NC_ERR_INVALID_ARG, "cache length %d + T=%d exceeds t_max %d", pos0, T, c->t_max);
  NC_CHECK(T == 1 || pos0 == 0 || m->adt != NC_F32, NC_ERR_UNSUPPORTED,
           "continuing a prefill needs a 16-bit model");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = prefill_common(m, tokens, B, T, c, s, pos0);
  if (st != NC_OK) return st;
  return run_lm_head(m, m->xn, (int64_t)B * T, logits, s);
}

nc_status nc_prefill_last(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                          float* logits_last, int32_t* argmax_out, nc_kv_cache* c, void* stream) {
  nc_status st = check_prefill_args(m, tokens, B, T, c);
  if (st != NC_OK) return st;
  NC_CHECK(!logits_last || aligned16(logits_last), NC_ERR_INVALID_ARG, "logits misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = prefill_common(m, tokens, B, T, c, s);
  if (st != NC_OK) return st;
  {
    ProfScope ps(m, NC_K_NORM, s);
    nc::launch_gather_rows(m->x, m->xl, B, T, m->cfg.d_model, s);
    nc::launch_rmsnorm(m->xl, m->xnl, m->adt, B, m->cfg.d_model, m->cfg.rms_eps, s);
  }
  float* lg = logits_last ? logits_last : m->logits_tmp;
  st = run_lm_head(m, m->xnl, B, lg, s);
  if (st != NC_OK) return st;
  if (argmax_out) {
    ProfScope ps(m, NC_K_ARGMAX, s);
    nc::launch_argmax(lg, B, m->cfg.vocab, argmax_out, s);
  }
  return check_launch();
}

nc_status nc_prefill_loss(nc_model* m, const int32_t* tokens, const int32_t* targets, int32_t B,
                          int32_t T, float* loss, float* mean, nc_kv_cache* c, void* stream) {
  nc_status st = check_prefill_args(m, tokens, B, T, c);
  if (st != NC_OK) return st;
  NC_CHECK(targets && mean, NC_ERR_INVALID_ARG, "NULL targets or mean");
  NC_CHECK((reinterpret_cast<uintptr_t>(targets) & 3u) == 0 &&
               (!loss || (reinterpret_cast<uintptr_t>(loss) & 3u) == 0) &&
               (reinterpret_cast<uintptr_t>(mean) & 3u) == 0,
           NC_ERR_INVALID_ARG, "targets, loss and mean must be 4-byte aligned");
  NC_CHECK(m->adt != NC_F32, NC_ERR_UNSUPPORTED,
           "the fused loss runs on the tensor-core path (16-bit activations)");
  const int64_t M = (int64_t)B * T;
  const int nblk = nc::lm_loss_blocks(m->cfg.vocab);
  const size_t b_part = round_up((size_t)M * nblk * sizeof(float2), 256),
               b_row = round_up((size_t)M * sizeof(float), 256);
  if (b_part + 2 * b_row > m->ce_ws_bytes) {
    cudaFree(m->ce_ws);
    m->ce_ws = nullptr;
    m->ce_ws_bytes = 0;
    if (cudaMalloc(&m->ce_ws, b_part + 2 * b_row) != cudaSuccess) {
      cudaGetLastError();
      m->ce_ws = nullptr;
      set_err("loss scratch allocation of %zu bytes failed", b_part + 2 * b_row);
      return NC_ERR_OOM;
    }
    m->ce_ws_bytes = b_part + 2 * b_row;
  }
  char* ws = static_cast<char*>(m->ce_ws);
  float2* part = reinterpret_cast<float2*>(ws);
  float* zt = reinterpret_cast<float*>(ws + b_part);
  float* rows = loss ? loss : reinterpret_cast<float*>(ws + b_part + b_row);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = prefill_common(m, tokens, B, T, c, s);
  if (st != NC_OK) return st;
  {
    ProfScope ps(m, NC_K_LM_HEAD, s);
    st = nc::tc_lm_loss(m->tc, m->xn, M, targets, part, zt, s);
    if (st != NC_OK) return st;
    nc::launch_ce_finish(part, nblk, zt, targets, m->cfg.vocab, M, rows, mean, m->status, s);
  }
  return check_launch();
}

nc_status nc_decode_step(nc_model* m, const int32_t* tokens, int32_t B, int32_t pos,
                         float* logits, int32_t* argmax_out, nc_kv_cache* c, void* stream) {
  NC_CHECK(m && c && tokens, NC_ERR_INVALID_ARG, "NULL model, cache or tokens");
  NC_CHECK(c->model == m, NC_ERR_INVALID_ARG, "cache belongs to another model");
  NC_CHECK(logits || argmax_out, NC_ERR_INVALID_ARG, "need logits or argmax_out");
  NC_CHECK(!logits || aligned16(logits), NC_ERR_INVALID_ARG, "logits misaligned");
  NC_CHECK(B >= 1 && B <= c->batch && B <= m->cfg.max_batch, NC_ERR_INVALID_ARG,
           "B=%d out of range", B);
  NC_CHECK(lens_equal(c, B, pos), NC_ERR_INVALID_ARG,
           "pos %d must equal the cache length of each of the %d sequences", pos, B);
  NC_CHECK(pos >= 1, NC_ERR_INVALID_ARG, "decode needs a prefilled cache (pos >= 1)");
  NC_CHECK(pos + 1 <= c->t_max, NC_ERR_INVALID_ARG, "cache full (t_max %d)", c->t_max);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool fused_ok = decode_fused_applies(m);
  NC_CHECK(fused_ok || m->decode_path != NC_DECODE_PERSISTENT, NC_ERR_UNSUPPORTED,
           "the persistent decode step does not support this shape");
  if (fused_ok && m->decode_path != NC_DECODE_KERNELS) {
    const std::vector<int32_t> pv(B, pos);
    nc_status st = decode_fused(m, tokens, B, pv.data(), logits, argmax_out, c, s);
    if (st == NC_OK) set_lens(c, B, pos + 1);
    return st;
  }
  {
    ProfScope ps(m, NC_K_EMBED, s);
    nc::launch_embed_norm(tokens, m->wte, m->cfg.dtype, m->x, m->xn, m->adt, B, m->cfg.d_model,
                          m->cfg.vocab, m->cfg.rms_eps, m->status, s);
  }
  nc_status st = run_blocks(m, c, B, 1, pos, s);
  if (st != NC_OK) return st;
  float* lg = logits ? logits : m->logits_tmp;
  st = run_lm_head(m, m->xn, B, lg, s);
  if (st != NC_OK) return st;
  if (argmax_out) {
    ProfScope ps(m, NC_K_ARGMAX, s);
    nc::launch_argmax(lg, B, m->cfg.vocab, argmax_out, s);
  }
  st = check_launch();
  if (st == NC_OK) set_lens(c, B, pos + 1);
  return st;
}

nc_status nc_decode_step_sample(nc_model* m, const int32_t* tokens, int32_t B, int32_t pos,
                                float temperature, const float* u, int32_t* next_out,
                                float* logits, nc_kv_cache* c, void* stream) {
  NC_CHECK(m && c && tokens && next_out, NC_ERR_INVALID_ARG, "NULL model, cache, tokens or next_out");
  NC_CHECK(c->model == m, NC_ERR_INVALID_ARG, "cache belongs to another model");
  NC_CHECK(!(temperature > 0.f) || u, NC_ERR_INVALID_ARG, "sampling at temperature %g needs u",
           (double)temperature);
  NC_CHECK(!logits || aligned16(logits), NC_ERR_INVALID_ARG, "logits misaligned");
  NC_CHECK(B >= 1 && B <= c->batch && B <= m->cfg.max_batch, NC_ERR_INVALID_ARG,
           "B=%d out of range", B);
  NC_CHECK(lens_equal(c, B, pos), NC_ERR_INVALID_ARG,
           "pos %d must equal the cache length of each of the %d sequences", pos, B);
  NC_CHECK(pos >= 1, NC_ERR_INVALID_ARG, "decode needs a prefilled cache (pos >= 1)");
  NC_CHECK(pos + 1 <= c->t_max, NC_ERR_INVALID_ARG, "cache full (t_max %d)", c->t_max);
  NC_CHECK(decode_fused_applies(m) && m->decode_path != NC_DECODE_KERNELS, NC_ERR_UNSUPPORTED,
           "sampling inside the step needs the persistent decode step (16-bit model of a "
           "supported shape)");
  nc_status st = decode_fused_init(m, static_cast<cudaStream_t>(stream));
  if (st != NC_OK) return st;
  const int groups = (m->dlay.vpad + 127) / 128;
  NC_CHECK(m->sms <= nc::dec::kMaxAttnBlocks &&
               (groups + m->sms - 1) / m->sms <= nc::dec::kMaxResidentGroups,
           NC_ERR_UNSUPPORTED, "vocabulary of %d too large to keep on chip for the draw",
           m->cfg.vocab);
  StepSample smp;
  smp.on = true;
  smp.temperature = temperature;
  smp.u = u;
  const std::vector<int32_t> pv(B, pos);
  st = decode_fused(m, tokens, B, pv.data(), logits, next_out, c, static_cast<cudaStream_t>(stream),
                    smp);
  if (st == NC_OK) set_lens(c, B, pos + 1);
  return st;
}

nc_status nc_generate_host_sample(nc_model* m, const int32_t* prompt, int32_t B, int32_t T,
                                  int32_t steps, float temperature, const float* u,
                                  int32_t* out_tokens, nc_kv_cache* c, void* stream) {
  NC_CHECK(m && c && prompt && out_tokens, NC_ERR_INVALID_ARG, "NULL argument");
  NC_CHECK(!(temperature > 0.f) || u, NC_ERR_INVALID_ARG, "sampling needs u");
  NC_CHECK(steps >= 0 && T + steps <= c->t_max && steps + 1 <= m->cfg.max_seq,
           NC_ERR_INVALID_ARG, "T + steps exceeds the cache (t_max %d)", c->t_max);
  nc_status st = check_prefill_args(m, m->tok_dev, B, T, c);
  if (st != NC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  NC_CUDA(cudaMemcpyAsync(m->tok_dev, prompt, sizeof(int32_t) * B * T, cudaMemcpyHostToDevice, s));
  if (temperature > 0.f)
    NC_CUDA(cudaMemcpyAsync(m->gen_u, u, sizeof(float) * B * (steps + 1), cudaMemcpyHostToDevice,
                            s));
  set_lens(c, c->batch, 0);
  st = nc_prefill_last(m, m->tok_dev, B, T, m->logits_tmp, nullptr, c, stream);
  if (st != NC_OK) return st;
  {
    ProfScope ps(m, NC_K_ARGMAX, s);
    nc::launch_sample(m->logits_tmp, B, m->cfg.vocab, temperature, m->gen_u, m->gen_dev, s);
  }
  for (int j = 0; j < steps; ++j) {
    st = nc_decode_step_sample(m, m->gen_dev + (size_t)j * B, B, T + j, temperature,
                               m->gen_u + (size_t)(j + 1) * B, m->gen_dev + (size_t)(j + 1) * B,
                               nullptr, c, stream);
    if (st != NC_OK) return st;
  }
  NC_CUDA(cudaMemcpyAsync(out_tokens, m->gen_dev, sizeof(int32_t) * B * (steps + 1),
                          cudaMemcpyDeviceToHost, s));
  NC_CUDA(cudaStreamSynchronize(s));
  return NC_OK;
}

nc_status nc_decode_step_ragged(nc_model* m, const int32_t* tokens, const int32_t* pos, int32_t B,
                                float* logits, int32_t* argmax_out, nc_kv_cache* c, void* stream) {
  NC_CHECK(m && c && tokens && pos, NC_ERR_INVALID_ARG, "NULL model, cache, tokens or positions");
  NC_CHECK(c->model == m, NC_ERR_INVALID_ARG, "cache belongs to another model");
  NC_CHECK(logits || argmax_out, NC_ERR_INVALID_ARG, "need logits or argmax_out");
  NC_CHECK(!logits || aligned16(logits), NC_ERR_INVALID_ARG, "logits misaligned");
  NC_CHECK(B >= 1 && B <= c->batch && B <= m->cfg.max_batch, NC_ERR_INVALID_ARG,
           "B=%d out of range", B);
  for (int32_t b = 0; b < B; ++b) {
    NC_CHECK(pos[b] == c->lens[b], NC_ERR_INVALID_ARG,
             "pos[%d] = %d must equal that sequence's cache length %d", b, pos[b], c->lens[b]);
    NC_CHECK(pos[b] >= 1, NC_ERR_INVALID_ARG, "sequence %d: decode needs a prefilled cache", b);
    NC_CHECK(pos[b] + 1 <= c->t_max, NC_ERR_INVALID_ARG, "sequence %d: cache full (t_max %d)", b,
             c->t_max);
  }
  NC_CHECK(decode_fused_applies(m) && m->decode_path != NC_DECODE_KERNELS, NC_ERR_UNSUPPORTED,
           "per-sequence positions need the persistent decode step (16-bit model of a supported "
           "shape)");
  nc_status st = decode_fused(m, tokens, B, pos, logits, argmax_out, c,
                              static_cast<cudaStream_t>(stream));
  if (st != NC_OK) return st;
  for (int32_t b = 0; b < B; ++b) c->lens[b] = pos[b] + 1;
  c->len = *std::max_element(c->lens.begin(), c->lens.end());
  return NC_OK;
}

nc_status nc_generate_host(nc_model* m, const int32_t* prompt, int32_t B, int32_t T,
                           int32_t steps, int32_t* out_tokens, nc_kv_cache* c, void* stream) {
  NC_CHECK(m && c && prompt && out_tokens, NC_ERR_INVALID_ARG, "NULL argument");
  NC_CHECK(steps >= 0 && T + steps <= c->t_max && steps + 1 <= m->cfg.max_seq,
           NC_ERR_INVALID_ARG, "T + steps exceeds the cache (t_max %d)", c->t_max);
  nc_status st = check_prefill_args(m, m->tok_dev, B, T, c);
  if (st != NC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  NC_CUDA(cudaMemcpyAsync(m->tok_dev, prompt, sizeof(int32_t) * B * T, cudaMemcpyHostToDevice, s));
  set_lens(c, c->batch, 0);
  st = nc_prefill_last(m, m->tok_dev, B, T, nullptr, m->gen_dev, c, stream);
  if (st != NC_OK) return st;
  for (int j = 0; j < steps; ++j) {
    st = nc_decode_step(m, m->gen_dev + (size_t)j * B, B, T + j, nullptr,
                        m->gen_dev + (size_t)(j + 1) * B, c, stream);
    if (st != NC_OK) return st;
  }
  NC_CUDA(cudaMemcpyAsync(out_tokens, m->gen_dev, sizeof(int32_t) * B * (steps + 1),
                          cudaMemcpyDeviceToHost, s));
  NC_CUDA(cudaStreamSynchronize(s));
  return NC_OK;
}

nc_status nc_decode_trace(nc_model* m, uint64_t* dev_buf, int32_t capacity) {
  NC_CHECK(m, NC_ERR_INVALID_ARG, "model is NULL");
  NC_CHECK(!dev_buf || capacity > 0, NC_ERR_INVALID_ARG, "capacity must be positive");
  m->dec_trace = reinterpret_cast<unsigned long long*>(dev_buf);
  m->dec_trace_cap = dev_buf ? capacity : 0;
  return NC_OK;
}

int32_t nc_decode_trace_entries(const nc_config* cfg) {
  return cfg ? nc::dec::trace_entries(cfg->n_layer) : 0;
}

nc_status nc_model_set_decode_path(nc_model* m, nc_decode_path path) {
  NC_CHECK(m, NC_ERR_INVALID_ARG, "model is NULL");
  NC_CHECK(path == NC_DECODE_AUTO || path == NC_DECODE_PERSISTENT || path == NC_DECODE_KERNELS,
           NC_ERR_INVALID_ARG, "unknown decode path %d", (int)path);
  m->decode_path = path;
  return NC_OK;
}

nc_status nc_kv_cache_set_length(nc_kv_cache* c, int32_t len) {
  NC_CHECK(c, NC_ERR_INVALID_ARG, "cache is NULL");
  NC_CHECK(len >= 0 && len <= c->len, NC_ERR_INVALID_ARG, "length %d outside [0, %d]", len, c->len);
  for (auto& l : c->lens) l = std::min(l, len);
  c->len = *std::max_element(c->lens.begin(), c->lens.end());
  return NC_OK;
}

nc_status nc_kv_cache_set_lengths(nc_kv_cache* c, const int32_t* lens, int32_t n) {
  NC_CHECK(c && lens, NC_ERR_INVALID_ARG, "NULL cache or lengths");
  NC_CHECK(n >= 1 && n <= c->batch, NC_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, c->batch);
  for (int32_t b = 0; b < n; ++b)
    NC_CHECK(lens[b] >= 0 && lens[b] <= c->lens[b], NC_ERR_INVALID_ARG,
             "sequence %d: length %d outside [0, %d]", b, lens[b], c->lens[b]);
  for (int32_t b = 0; b < n; ++b) c->lens[b] = lens[b];
  c->len = *std::max_element(c->lens.begin(), c->lens.end());
  return NC_OK;
}

nc_status nc_kv_cache_lengths(const nc_kv_cache* c, int32_t* lens, int32_t n) {
  NC_CHECK(c && lens, NC_ERR_INVALID_ARG, "NULL cache or output");
  NC_CHECK(n >= 1 && n <= c->batch, NC_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, c->batch);
  for (int32_t b = 0; b < n; ++b) lens[b] = c->lens[b];
  return NC_OK;
}

nc_status nc_profile_begin(nc_model* m) {
  NC_CHECK(m, NC_ERR_INVALID_ARG, "model is NULL");
  m->prof = true;
  return NC_OK;
}

nc_status nc_profile_end(nc_model* m, void* stream, nc_kernel_time* out) {
  NC_CHECK(m && out, NC_ERR_INVALID_ARG, "NULL argument");
  NC_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  for (int k = 0; k < NC_K_COUNT; ++k) out[k] = nc_kernel_time{0.0, 0};
  for (auto& r : m->recs) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    out[r.kind].ms += ms;
    out[r.kind].launches += r.launches;
    m->event_pool.push_back(r.a);
    m->event_pool.push_back(r.b);
  }
  m->recs.clear();
  m->prof = false;
  return NC_OK;
}

int64_t nc_launch_count(void) { return g_launches.load(); }

nc_status nc_model_check(nc_model* m, void* stream) {
  NC_CHECK(m, NC_ERR_INVALID_ARG, "model is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  NC_CUDA(cudaStreamSynchronize(s));
  NC_CUDA(cudaMemcpy(&word, m->status, 4, cudaMemcpyDeviceToHost));
  NC_CUDA(cudaMemset(m->status, 0, 4));
  if (word & nc::ST_TIMEOUT) {
    // a persistent step gave up: clear its abort word and barrier counter
    NC_CUDA(cudaMemset(m->status + 1, 0, 4));
    if (m->d_bar) NC_CUDA(cudaMemset(m->d_bar, 0, 8));
    m->bar_base = 0;
    set_err("a kernel's bounded wait timed out (status 0x%x)", word);
    return NC_ERR_DEVICE_TIMEOUT;
  }
  if (word & nc::ST_BAD_TOKEN) {
    set_err("a token id was outside [0, vocab) (an input token: row 0 was used; a loss "
            "target: the row was left out)");
    return NC_ERR_BOUNDS;
  }
  if (word & nc::ST_RANGE) {
    set_err("a value stored in fp16 exceeded its range (|v| >= 65520) and became inf; "
            "act_dtype NC_BF16 has fp32's range");
    return NC_ERR_RANGE;
  }
  return NC_OK;
}

// ------------------------------------------------------------ single steps
nc_status nc_op_rmsnorm(const float* x, void* y, nc_dtype y_dtype, int64_t M, int32_t d,
                        float eps, void* stream) {
  NC_CHECK(x && y && aligned16(x) && aligned16(y), NC_ERR_INVALID_ARG, "NULL/misaligned");
  NC_CHECK(M >= 0 && d > 0 && d % 4 == 0, NC_ERR_INVALID_ARG, "d must be a positive multiple of 4");
  NC_CHECK(y_dtype == NC_F32 || y_dtype == NC_BF16 || y_dtype == NC_F16, NC_ERR_INVALID_ARG,
           "bad dtype");
  if (M == 0) return NC_OK;
  nc::launch_rmsnorm(x, y, y_dtype, M, d, eps, static_cast<cudaStream_t>(stream));
  return check_launch();
}

nc_status nc_op_gemm(const void* A, const void* B, float* C, int32_t M, int32_t N, int32_t K,
                     nc_dtype dtype, void* stream) {
  NC_CHECK(A && B && C && aligned16(A) && aligned16(B) && aligned16(C), NC_ERR_INVALID_ARG,
           "NULL/misaligned");
  NC_CHECK(M >= 0 && N > 0 && K > 0, NC_ERR_INVALID_ARG, "bad sizes");
  if (M == 0) return NC_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == NC_BF16 || dtype == NC_F16) {
    NC_CHECK(K % 64 == 0 && N % 16 == 0, NC_ERR_UNSUPPORTED, "16-bit GEMM needs K%%64==0, N%%16==0");
    return nc::tc_gemm_f32out(A, B, C, M, N, K, dtype, s);
  }
  NC_CHECK(dtype == NC_F32, NC_ERR_INVALID_ARG, "bad dtype");
  nc::launch_gemm_simt(A, B, C, M, N, K, N, dtype, s);
  return check_launch();
}

nc_status nc_op_quantize_e4m3(const void* x, nc_dtype dtype, int64_t rows, int32_t cols, uint8_t* q,
                              float* scale, void* stream) {
  NC_CHECK(x && q && scale && aligned16(x) && aligned16(q), NC_ERR_INVALID_ARG, "NULL/misaligned");
  NC_CHECK(rows >= 0 && rows <= INT32_MAX && cols > 0 && cols % 16 == 0, NC_ERR_INVALID_ARG,
           "bad sizes");
  NC_CHECK(dtype == NC_F32 || dtype == NC_BF16 || dtype == NC_F16, NC_ERR_INVALID_ARG, "bad dtype");
  return nc::quantize_e4m3(x, dtype, rows, cols, q, scale, static_cast<cudaStream_t>(stream));
}

size_t nc_op_cross_entropy_scratch_bytes(int32_t M, int32_t N) {
  if (M < 0 || N <= 0) return 0;
  return round_up((size_t)M * nc::lm_loss_blocks(N) * sizeof(float2), 256) +
         2 * round_up((size_t)M * sizeof(float), 256);
}

nc_status nc_op_cross_entropy(const void* A, const void* B, const int32_t* targets, int32_t M,
                              int32_t N, int32_t K, nc_dtype dtype, float* loss, float* mean,
                              void* scratch, size_t scratch_bytes, void* stream) {
  NC_CHECK(A && B && targets && mean && scratch && aligned16(A) && aligned16(B) &&
               aligned16(scratch) && (reinterpret_cast<uintptr_t>(targets) & 3u) == 0 &&
               (!loss || (reinterpret_cast<uintptr_t>(loss) & 3u) == 0) &&
               (reinterpret_cast<uintptr_t>(mean) & 3u) == 0,
           NC_ERR_INVALID_ARG, "NULL/misaligned");
  NC_CHECK(M >= 0 && N > 0 && K > 0, NC_ERR_INVALID_ARG, "bad sizes");
  NC_CHECK(dtype == NC_BF16 || dtype == NC_F16, NC_ERR_INVALID_ARG, "dtype must be NC_BF16 or NC_F16");
  NC_CHECK(K % 64 == 0, NC_ERR_UNSUPPORTED, "needs K%%64==0");
  NC_CHECK(scratch_bytes >= nc_op_cross_entropy_scratch_bytes(M, N), NC_ERR_INVALID_ARG,
           "scratch too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t b_part = round_up((size_t)M * nc::lm_loss_blocks(N) * sizeof(float2), 256),
               b_row = round_up((size_t)M * sizeof(float), 256);
  char* ws = static_cast<char*>(scratch);
  float2* part = reinterpret_cast<float2*>(ws);
  float* zt = reinterpret_cast<float*>(ws + b_part);
  float* rows = loss ? loss : reinterpret_cast<float*>(ws + b_part + b_row);
  if (M > 0) {
    nc_status st = nc::tc_cross_entropy(A, B, targets, M, N, K, dtype, part, zt, s);
    if (st != NC_OK) return st;
  }
  nc::launch_ce_finish(part, nc::lm_loss_blocks(N), zt, targets, N, M, rows, mean, nullptr, s);
  return check_launch();
}

size_t nc_op_gemv_e4m3_scratch_bytes(int32_t N, int32_t K, int32_t B) {
  if (N <= 0 || K <= 0 || B <= 0 || B > 128) return 0;
  return nc::gemv_e4m3_scratch_bytes(N, K, B);
}

nc_status nc_op_gemv_e4m3(const uint8_t* wq, const float* w_scale, int32_t N, int32_t K,
                          const float* x, int32_t B, float* y, void* scratch, size_t scratch_bytes,
                          void* stream) {
  NC_CHECK(wq && w_scale && x && y && scratch && aligned16(wq) && aligned16(x) && aligned16(y) &&
               aligned16(scratch),
           NC_ERR_INVALID_ARG, "NULL/misaligned");
  NC_CHECK(N > 0 && K > 0 && K % 128 == 0 && B >= 1 && B <= 128, NC_ERR_INVALID_ARG, "bad sizes");
  NC_CHECK(scratch_bytes >= nc::gemv_e4m3_scratch_bytes(N, K, B), NC_ERR_INVALID_ARG,
           "scratch too small");
  return nc::gemv_e4m3(wq, w_scale, N, K, x, B, y, scratch, static_cast<cudaStream_t>(stream));
}

nc_status nc_op_attention_prefill(const void* q, const void* k, const void* v, void* o, int32_t B,
                                  int32_t H, int32_t Hkv, int32_t T, int32_t t_max, int32_t hd,
                                  nc_dtype dtype, void* stream) {
  NC_CHECK(q && k && v && o && aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o),
           NC_ERR_INVALID_ARG, "NULL/misaligned");
  NC_CHECK(B > 0 && H > 0 && Hkv > 0 && H % Hkv == 0 && T > 0 && T <= t_max && hd > 0 &&
               hd % 2 == 0 && hd <= 128,
           NC_ERR_INVALID_ARG, "bad sizes");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == NC_BF16 || dtype == NC_F16) {
    NC_CHECK(hd == 128, NC_ERR_UNSUPPORTED, "16-bit attention needs head_dim 128");
    const int64_t one_layer = (int64_t)B * Hkv * t_max * hd;
    nc_status st = nc::tc_attention_prefill_tc(q, k, v, o, B, H, Hkv, T, 0, t_max, 1, one_layer,
                                               0, dtype, nullptr, s);
    if (st == NC_OK) return NC_OK;
    return nc::tc_attention_prefill(q, k, v, o, B, H, Hkv, T, t_max, dtype, s);
  }
  NC_CHECK(dtype == NC_F32, NC_ERR_INVALID_ARG, "bad dtype");
  nc::launch_attention_prefill_simt(q, k, v, o, B, H, Hkv, T, t_max, hd, dtype, s);
  return check_launch();
}

size_t nc_op_attention_decode_scratch_bytes(int32_t B, int32_t H, int32_t t_max, int32_t hd) {
  if (B <= 0 || H <= 0 || t_max <= 0 || hd <= 0) return 0;
  const int ns = std::min(64, (t_max + 63) / 64);   // the most splits any call can use
  return (size_t)B * H * ns * (hd + 2) * sizeof(float);
}

nc_status nc_op_attention_decode(const void* q, const void* k, const void* v, void* o, int32_t B,
                                 int32_t H, int32_t Hkv, int32_t len, int32_t t_max, int32_t hd,
                                 nc_dtype dtype, void* scratch, size_t scratch_bytes,
                                 void* stream) {
  NC_CHECK(q && k && v && o && scratch, NC_ERR_INVALID_ARG, "NULL pointer");
  NC_CHECK(B > 0 && H > 0 && Hkv > 0 && H % Hkv == 0 && len > 0 && len <= t_max && hd > 0 &&
               hd % 2 == 0 && hd <= 128,
           NC_ERR_INVALID_ARG, "bad sizes");
  NC_CHECK(dtype == NC_F32 || dtype == NC_BF16 || dtype == NC_F16, NC_ERR_INVALID_ARG, "bad dtype");
  NC_CHECK(scratch_bytes >= nc::decode_attention_scratch_bytes(B, H, Hkv, len, hd),
           NC_ERR_INVALID_ARG, "scratch too small");
  nc::launch_attention_decode(q, k, v, o, B, H, Hkv, len, t_max, hd, dtype,
                              static_cast<float*>(scratch), static_cast<cudaStream_t>(stream));
  return check_launch();
}

nc_status nc_op_argmax(const float* x, int32_t rows, int32_t n, int32_t* out, void* stream) {
  NC_CHECK(x && out, NC_ERR_INVALID_ARG, "NULL pointer");
  NC_CHECK(rows >= 0 && n > 0, NC_ERR_INVALID_ARG, "bad sizes");
  if (rows == 0) return NC_OK;
  nc::launch_argmax(x, rows, n, out, static_cast<cudaStream_t>(stream));
  return check_launch();
}

nc_status nc_op_sample(const float* logits, int32_t rows, int32_t n, float temperature,
                       const float* u, int32_t* out, void* stream) {
  NC_CHECK(logits && u && out, NC_ERR_INVALID_ARG, "NULL pointer");
  NC_CHECK(rows >= 0 && n > 0, NC_ERR_INVALID_ARG, "bad sizes");
  if (rows == 0) return NC_OK;
  nc::launch_sample(logits, rows, n, temperature, u, out, static_cast<cudaStream_t>(stream));
  return check_launch();
}

}  // extern "C"
