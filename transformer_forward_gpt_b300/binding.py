"""ctypes binding of libnc.so (include/nc.h), same entry-point names.

Argument marshalling only: torch tensors are passed as their device pointers,
streams as their cudaStream_t handle; every step of the forward pass runs in the
library's CUDA kernels. A missing or unloadable library raises at import of the
first call -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnc.so")

NC_OK, NC_ERR_INVALID_ARG, NC_ERR_UNSUPPORTED, NC_ERR_OOM, NC_ERR_CUDA, \
    NC_ERR_DEVICE_TIMEOUT, NC_ERR_BOUNDS, NC_ERR_RANGE = range(8)
NC_F32, NC_BF16, NC_F16 = 0, 1, 2

EXPORTS = (
    "nc_version", "nc_status_string", "nc_last_error", "nc_param_count", "nc_model_create",
    "nc_model_destroy", "nc_kv_cache_bytes", "nc_kv_cache_alloc", "nc_kv_cache_view",
    "nc_kv_cache_free", "nc_prefill", "nc_prefill_last", "nc_decode_step", "nc_generate_host",
    "nc_model_check", "nc_op_rmsnorm", "nc_op_gemm", "nc_op_attention_prefill",
    "nc_op_attention_decode_scratch_bytes", "nc_op_attention_decode", "nc_op_argmax",
    "nc_kv_cache_set_length", "nc_profile_begin", "nc_profile_end", "nc_launch_count",
    "nc_op_attention_decode_noalloc", "nc_model_set_decode_path", "nc_decode_trace",
    "nc_decode_trace_entries", "nc_op_sample", "nc_prefill_continue",
    "nc_decode_step_ragged", "nc_kv_cache_set_lengths", "nc_kv_cache_lengths",
    "nc_decode_step_sample", "nc_generate_host_sample", "nc_op_quantize_e4m3",
    "nc_prefill_loss", "nc_op_cross_entropy_scratch_bytes", "nc_op_cross_entropy",
    "nc_op_gemv_e4m3_scratch_bytes", "nc_op_gemv_e4m3",
)

KERNEL_KINDS = ("embed", "norm", "qkv", "attn_prefill", "attn_decode", "oproj", "fc", "proj",
                "lm_head", "argmax", "decode_step")


class NcConfig(C.Structure):
    _fields_ = [("vocab", C.c_int32), ("d_model", C.c_int32), ("n_layer", C.c_int32),
                ("n_head", C.c_int32), ("n_kv_head", C.c_int32), ("head_dim", C.c_int32),
                ("d_mlp", C.c_int32), ("rope_base", C.c_float), ("rms_eps", C.c_float),
                ("max_seq", C.c_int32), ("max_batch", C.c_int32), ("dtype", C.c_int),
                ("act_dtype", C.c_int)]


class NcKernelTime(C.Structure):
    _fields_ = [("ms", C.c_double), ("launches", C.c_int64)]


class NcWeights(C.Structure):
    _fields_ = [("wte", C.c_void_p), ("lm_head", C.c_void_p),
                ("wq", C.POINTER(C.c_void_p)), ("wk", C.POINTER(C.c_void_p)),
                ("wv", C.POINTER(C.c_void_p)), ("wo", C.POINTER(C.c_void_p)),
                ("w_fc", C.POINTER(C.c_void_p)), ("w_proj", C.POINTER(C.c_void_p))]


_lib = None


def load(path: str = LIB_PATH):
    """Loads libnc.so once; raises OSError/RuntimeError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m transformer_forward_gpt_b300.build`")
    lib = C.CDLL(path)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "nc_version": (C.c_char_p, []),
        "nc_status_string": (C.c_char_p, [C.c_int]),
        "nc_last_error": (C.c_char_p, []),
        "nc_param_count": (i64, [C.POINTER(NcConfig)]),
        "nc_model_create": (C.c_int, [C.POINTER(NcConfig), C.POINTER(NcWeights), C.POINTER(vp)]),
        "nc_model_destroy": (None, [vp]),
        "nc_kv_cache_bytes": (sz, [C.POINTER(NcConfig), i32, i32]),
        "nc_kv_cache_alloc": (C.c_int, [vp, i32, i32, vp, C.POINTER(vp)]),
        "nc_kv_cache_view": (C.c_int, [vp, C.POINTER(vp), C.POINTER(vp), C.POINTER(i32),
                                       C.POINTER(i32), C.POINTER(i32)]),
        "nc_kv_cache_free": (None, [vp]),
        "nc_prefill": (C.c_int, [vp, vp, i32, i32, vp, vp, vp]),
        "nc_prefill_continue": (C.c_int, [vp, vp, i32, i32, vp, vp, vp]),
        "nc_prefill_last": (C.c_int, [vp, vp, i32, i32, vp, vp, vp, vp]),
        "nc_prefill_loss": (C.c_int, [vp, vp, vp, i32, i32, vp, vp, vp, vp]),
        "nc_op_cross_entropy_scratch_bytes": (C.c_size_t, [i32, i32]),
        "nc_op_cross_entropy": (C.c_int, [vp, vp, vp, i32, i32, i32, C.c_int, vp, vp, vp,
                                          C.c_size_t, vp]),
        "nc_decode_step": (C.c_int, [vp, vp, i32, i32, vp, vp, vp, vp]),
        "nc_generate_host": (C.c_int, [vp, vp, i32, i32, i32, vp, vp, vp]),
        "nc_model_check": (C.c_int, [vp, vp]),
        "nc_op_rmsnorm": (C.c_int, [vp, vp, C.c_int, i64, i32, C.c_float, vp]),
        "nc_op_gemm": (C.c_int, [vp, vp, vp, i32, i32, i32, C.c_int, vp]),
        "nc_op_attention_prefill": (C.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                              C.c_int, vp]),
        "nc_op_attention_decode_scratch_bytes": (sz, [i32, i32, i32, i32]),
        "nc_op_attention_decode": (C.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                             C.c_int, vp, sz, vp]),
        "nc_op_argmax": (C.c_int, [vp, i32, i32, vp, vp]),
        "nc_op_sample": (C.c_int, [vp, i32, i32, C.c_float, vp, vp, vp]),
        "nc_op_quantize_e4m3": (C.c_int, [vp, C.c_int, i64, i32, vp, vp, vp]),
        "nc_op_gemv_e4m3_scratch_bytes": (sz, [i32, i32, i32]),
        "nc_op_gemv_e4m3": (C.c_int, [vp, vp, i32, i32, vp, i32, vp, vp, sz, vp]),
        "nc_kv_cache_set_length": (C.c_int, [vp, i32]),
        "nc_profile_begin": (C.c_int, [vp]),
        "nc_profile_end": (C.c_int, [vp, vp, C.POINTER(NcKernelTime)]),
        "nc_launch_count": (i64, []),
        "nc_op_attention_decode_noalloc": (C.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                     i32, C.c_int, vp]),
        "nc_model_set_decode_path": (C.c_int, [vp, C.c_int]),
        "nc_decode_trace": (C.c_int, [vp, vp, i32]),
        "nc_decode_trace_entries": (i32, [C.POINTER(NcConfig)]),
        "nc_decode_step_ragged": (C.c_int, [vp, vp, C.POINTER(i32), i32, vp, vp, vp, vp]),
        "nc_decode_step_sample": (C.c_int, [vp, vp, i32, i32, C.c_float, vp, vp, vp, vp, vp]),
        "nc_generate_host_sample": (C.c_int, [vp, vp, i32, i32, i32, C.c_float, vp, vp, vp, vp]),
        "nc_kv_cache_set_lengths": (C.c_int, [vp, C.POINTER(i32), i32]),
        "nc_kv_cache_lengths": (C.c_int, [vp, C.POINTER(i32), i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


class NcError(RuntimeError):
    def __init__(self, code, where):
        lib = load()
        super().__init__(f"{where}: {lib.nc_status_string(code).decode()} "
                         f"({lib.nc_last_error().decode()})")
        self.code = code


def _check(code, where):
    if code != NC_OK:
        raise NcError(code, where)


def _ptr(t):
    """Device pointer of a torch tensor (or None / int passthrough)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(shape, max_seq, max_batch, act_dtype=NC_F16) -> NcConfig:
    """Config of a synthetic shape: weights in the shape's dtype; the tensor-core
    path keeps activations / KV cache in `act_dtype` (fp16 by default)."""
    wdt = NC_BF16 if shape.dtype == "bf16" else NC_F32
    return NcConfig(shape.vocab, shape.d_model, shape.n_layer, shape.n_head, shape.n_kv_head,
                    shape.head_dim, shape.d_mlp, shape.rope_base, shape.rms_eps, max_seq,
                    max_batch, wdt, NC_F32 if wdt == NC_F32 else act_dtype)


# ------------------------------------------------------------ same-name calls
def nc_version():
    return load().nc_version().decode()


def nc_param_count(cfg: NcConfig) -> int:
    return load().nc_param_count(C.byref(cfg))


def nc_kv_cache_bytes(cfg: NcConfig, batch, t_max) -> int:
    return load().nc_kv_cache_bytes(C.byref(cfg), batch, t_max)


def nc_model_create(cfg: NcConfig, wte, lm_head, layers):
    """layers: list of (wq, wk, wv, wo, w_fc, w_proj) device tensors."""
    lib = load()
    L = cfg.n_layer
    arrs = [(C.c_void_p * L)(*[_ptr(layer[i]) for layer in layers]) for i in range(6)]
    w = NcWeights(_ptr(wte), _ptr(lm_head), *[C.cast(a, C.POINTER(C.c_void_p)) for a in arrs])
    out = C.c_void_p()
    _check(lib.nc_model_create(C.byref(cfg), C.byref(w), C.byref(out)), "nc_model_create")
    return out.value


def nc_model_destroy(model):
    load().nc_model_destroy(model)


def nc_kv_cache_alloc(model, batch, t_max, mem=None):
    out = C.c_void_p()
    _check(load().nc_kv_cache_alloc(model, batch, t_max, _ptr(mem), C.byref(out)),
           "nc_kv_cache_alloc")
    return out.value


def nc_kv_cache_view(cache):
    k, v = C.c_void_p(), C.c_void_p()
    ln, b, t = C.c_int32(), C.c_int32(), C.c_int32()
    _check(load().nc_kv_cache_view(cache, C.byref(k), C.byref(v), C.byref(ln), C.byref(b),
                                   C.byref(t)), "nc_kv_cache_view")
    return k.value, v.value, ln.value, b.value, t.value


def nc_kv_cache_free(cache):
    load().nc_kv_cache_free(cache)


def nc_prefill(model, tokens, B, T, logits, cache, stream=None):
    _check(load().nc_prefill(model, _ptr(tokens), B, T, _ptr(logits), cache, _stream(stream)),
           "nc_prefill")


def nc_prefill_continue(model, tokens, B, T, logits, cache, stream=None):
    _check(load().nc_prefill_continue(model, _ptr(tokens), B, T, _ptr(logits), cache,
                                      _stream(stream)), "nc_prefill_continue")


def nc_prefill_last(model, tokens, B, T, logits_last, argmax_out, cache, stream=None):
    _check(load().nc_prefill_last(model, _ptr(tokens), B, T, _ptr(logits_last), _ptr(argmax_out),
                                  cache, _stream(stream)), "nc_prefill_last")


def nc_op_cross_entropy_scratch_bytes(M, N):
    return load().nc_op_cross_entropy_scratch_bytes(M, N)


def nc_op_cross_entropy(A, B, targets, M, N, K, dtype, loss, mean, scratch, scratch_bytes,
                        stream=None):
    _check(load().nc_op_cross_entropy(_ptr(A), _ptr(B), _ptr(targets), M, N, K, dtype, _ptr(loss),
                                      _ptr(mean), _ptr(scratch), scratch_bytes, _stream(stream)),
           "nc_op_cross_entropy")


def nc_prefill_loss(model, tokens, targets, B, T, loss, mean, cache, stream=None):
    _check(load().nc_prefill_loss(model, _ptr(tokens), _ptr(targets), B, T, _ptr(loss), _ptr(mean),
                                  cache, _stream(stream)), "nc_prefill_loss")


def nc_decode_step(model, tokens, B, pos, logits, argmax_out, cache, stream=None):
    _check(load().nc_decode_step(model, _ptr(tokens), B, pos, _ptr(logits), _ptr(argmax_out),
                                 cache, _stream(stream)), "nc_decode_step")


NC_DECODE_AUTO, NC_DECODE_PERSISTENT, NC_DECODE_KERNELS = 0, 1, 2


def nc_model_set_decode_path(model, path):
    _check(load().nc_model_set_decode_path(model, path), "nc_model_set_decode_path")


def nc_decode_trace(model, buf):
    """buf: device uint64 (torch int64) tensor, or None to switch tracing off."""
    _check(load().nc_decode_trace(model, _ptr(buf), 0 if buf is None else buf.numel()),
           "nc_decode_trace")


def nc_decode_trace_entries(cfg):
    return load().nc_decode_trace_entries(C.byref(cfg))


def nc_generate_host(model, prompt, B, T, steps, out_tokens, cache, stream=None):
    """prompt / out_tokens: host int32 tensors (pinned for overlap); out is [steps+1, B]."""
    _check(load().nc_generate_host(model, _ptr(prompt), B, T, steps, _ptr(out_tokens), cache,
                                   _stream(stream)), "nc_generate_host")


def nc_model_check(model, stream=None):
    """Returns the status code (does not raise) after reading the device status word."""
    return load().nc_model_check(model, _stream(stream))


def nc_op_rmsnorm(x, y, y_dtype, M, d, eps, stream=None):
    _check(load().nc_op_rmsnorm(_ptr(x), _ptr(y), y_dtype, M, d, eps, _stream(stream)),
           "nc_op_rmsnorm")


def nc_op_gemm(A, B, Cout, M, N, K, dtype, stream=None):
    _check(load().nc_op_gemm(_ptr(A), _ptr(B), _ptr(Cout), M, N, K, dtype, _stream(stream)),
           "nc_op_gemm")


def nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, t_max, hd, dtype, stream=None):
    _check(load().nc_op_attention_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Hkv, T, t_max,
                                          hd, dtype, _stream(stream)), "nc_op_attention_prefill")


def nc_op_attention_decode_scratch_bytes(B, H, t_max, hd):
    return load().nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)


def nc_op_attention_decode(q, k, v, o, B, H, Hkv, length, t_max, hd, dtype, scratch,
                           scratch_bytes, stream=None):
    _check(load().nc_op_attention_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Hkv, length,
                                         t_max, hd, dtype, _ptr(scratch), scratch_bytes,
                                         _stream(stream)), "nc_op_attention_decode")


def nc_op_argmax(x, rows, n, out, stream=None):
    _check(load().nc_op_argmax(_ptr(x), rows, n, _ptr(out), _stream(stream)), "nc_op_argmax")


def nc_op_sample(logits, rows, n, temperature, u, out, stream=None):
    _check(load().nc_op_sample(_ptr(logits), rows, n, float(temperature), _ptr(u), _ptr(out),
                               _stream(stream)), "nc_op_sample")


def nc_op_quantize_e4m3(x, dtype, rows, cols, q, scale, stream=None):
    _check(load().nc_op_quantize_e4m3(_ptr(x), dtype, rows, cols, _ptr(q), _ptr(scale),
                                      _stream(stream)), "nc_op_quantize_e4m3")


def nc_op_gemv_e4m3_scratch_bytes(N, K, B):
    return load().nc_op_gemv_e4m3_scratch_bytes(N, K, B)


def nc_op_gemv_e4m3(wq, w_scale, N, K, x, B, y, scratch, scratch_bytes, stream=None):
    _check(load().nc_op_gemv_e4m3(_ptr(wq), _ptr(w_scale), N, K, _ptr(x), B, _ptr(y), _ptr(scratch),
                                  scratch_bytes, _stream(stream)), "nc_op_gemv_e4m3")


def nc_op_attention_decode_noalloc(q, k, v, o, B, H, Hkv, length, t_max, hd, dtype, stream=None):
    """Decode attention whose scratch is a fixed array inside the library (no allocation)."""
    _check(load().nc_op_attention_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Hkv,
                                                 length, t_max, hd, dtype, _stream(stream)),
           "nc_op_attention_decode_noalloc")


def nc_decode_step_ragged(model, tokens, pos, B, logits, argmax_out, cache, stream=None):
    """pos: host sequence of B positions (one per sequence)."""
    arr = (C.c_int32 * B)(*[int(x) for x in pos])
    _check(load().nc_decode_step_ragged(model, _ptr(tokens), arr, B, _ptr(logits), _ptr(argmax_out),
                                        cache, _stream(stream)), "nc_decode_step_ragged")


def nc_decode_step_sample(model, tokens, B, pos, temperature, u, next_out, logits, cache,
                          stream=None):
    _check(load().nc_decode_step_sample(model, _ptr(tokens), B, pos, float(temperature), _ptr(u),
                                        _ptr(next_out), _ptr(logits), cache, _stream(stream)),
           "nc_decode_step_sample")


def nc_generate_host_sample(model, prompt, B, T, steps, temperature, u, out_tokens, cache,
                            stream=None):
    """prompt: pinned/host int32 [B, T]; u: host float32 [steps + 1, B] (or None when greedy);
    out_tokens: host int32 [steps + 1, B]."""
    _check(load().nc_generate_host_sample(model, _ptr(prompt), B, T, steps, float(temperature),
                                          _ptr(u), _ptr(out_tokens), cache, _stream(stream)),
           "nc_generate_host_sample")


def nc_kv_cache_set_lengths(cache, lens):
    arr = (C.c_int32 * len(lens))(*[int(x) for x in lens])
    _check(load().nc_kv_cache_set_lengths(cache, arr, len(lens)), "nc_kv_cache_set_lengths")


def nc_kv_cache_lengths(cache, n):
    arr = (C.c_int32 * n)()
    _check(load().nc_kv_cache_lengths(cache, arr, n), "nc_kv_cache_lengths")
    return list(arr)


def nc_kv_cache_set_length(cache, length):
    _check(load().nc_kv_cache_set_length(cache, length), "nc_kv_cache_set_length")


def nc_profile_begin(model):
    _check(load().nc_profile_begin(model), "nc_profile_begin")


def nc_profile_end(model, stream=None):
    """{kind: (ms, launches)} of the intervals recorded since nc_profile_begin."""
    out = (NcKernelTime * len(KERNEL_KINDS))()
    _check(load().nc_profile_end(model, _stream(stream), out), "nc_profile_end")
    return {k: (out[i].ms, out[i].launches) for i, k in enumerate(KERNEL_KINDS)}


def nc_launch_count():
    return load().nc_launch_count()


# ----------------------------------------------------------------- helpers
class Model:
    """Owns device copies of one synthetic model's weights plus the nc_model.

    Marshalling only: weights are torch tensors on the device; every forward
    step runs in libnc.
    """

    def __init__(self, weights, max_seq, max_batch, device="cuda", act_dtype=NC_F16):
        import torch
        shape = weights.shape
        self.shape = shape
        self.cfg = make_config(shape, max_seq, max_batch, act_dtype)
        self.device = device

        def dev(name, arr):
            if shape.dtype == "bf16":
                bits = weights.bits[name]
                return torch.from_numpy(bits.view("int16")).view(torch.bfloat16).to(device)
            return torch.from_numpy(arr).to(device)
        self.wte = dev("wte", weights.wte)
        self.lm_head = dev("lm_head", weights.lm_head)
        names = ("wq", "wk", "wv", "wo", "w_fc", "w_proj")
        self.layers = [tuple(dev(f"layers.{l}.{n}", m) for n, m in zip(names, mats))
                       for l, mats in enumerate(weights.layers)]
        self.handle = nc_model_create(self.cfg, self.wte, self.lm_head, self.layers)

    def cache(self, batch, t_max):
        return KVCache(self, batch, t_max)

    def close(self):
        if self.handle:
            nc_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    def __init__(self, model: Model, batch, t_max):
        self.model = model
        self.handle = nc_kv_cache_alloc(model.handle, batch, t_max)
        self.batch, self.t_max = batch, t_max

    def tensors(self):
        """(k, v) torch views of shape [L, batch, Hkv, t_max, hd] (no copy)."""
        import torch
        s = self.model.shape
        kp, vp, _, _, _ = nc_kv_cache_view(self.handle)
        dt = {NC_BF16: torch.bfloat16, NC_F16: torch.float16,
              NC_F32: torch.float32}[self.model.cfg.act_dtype]
        n = s.n_layer * self.batch * s.n_kv_head * self.t_max * s.head_dim
        shp = (s.n_layer, self.batch, s.n_kv_head, self.t_max, s.head_dim)
        return tuple(_wrap_device(p, n, dt, self.model.device).view(shp) for p in (kp, vp))

    @property
    def length(self):
        return nc_kv_cache_view(self.handle)[2]

    def close(self):
        if self.handle:
            nc_kv_cache_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _wrap_device(ptr, numel, dtype, device):
    """A torch tensor aliasing library-owned device memory (kept alive by its owner)."""
    import torch
    esz = torch.tensor([], dtype=dtype).element_size()
    # torch has no public "from pointer" for CUDA; go through __cuda_array_interface__.
    class _Holder:
        __cuda_array_interface__ = {
            "shape": (numel,), "typestr": "<i2" if esz == 2 else "<f4",
            "data": (ptr, False), "version": 3,
        }
    t = torch.as_tensor(_Holder(), device=device)
    return t.view(dtype)
