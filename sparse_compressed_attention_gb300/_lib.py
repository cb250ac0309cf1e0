"""ctypes binding of libv4attn.so: the C ABI of include/v4attn.h, same names.

Argument marshalling only: tensors are checked for device, dtype, contiguity
and alignment, then their data pointers and the current CUDA stream are
handed to the library.  Every step of the path runs in the library's CUDA
kernels; there is no fallback.  A missing library raises at first use.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

V4_OK, V4_ERR_INVALID_ARG, V4_ERR_UNSUPPORTED, V4_ERR_WORKSPACE, V4_ERR_CUDA, \
    V4_ERR_TIMEOUT, V4_ERR_BAD_INDEX, V4_ERR_BOUND = range(8)
V4_F32, V4_BF16 = 0, 1
V4_PATH_AUTO, V4_PATH_SIMT, V4_PATH_TC = 0, 1, 2

STATUS_NAMES = {0: "V4_OK", 1: "V4_ERR_INVALID_ARG", 2: "V4_ERR_UNSUPPORTED", 3: "V4_ERR_WORKSPACE",
                4: "V4_ERR_CUDA", 5: "V4_ERR_TIMEOUT", 6: "V4_ERR_BAD_INDEX", 7: "V4_ERR_BOUND"}

# every symbol include/v4attn.h declares
EXPORTS = ["v4_rope_inv_freq", "v4_workspace_size", "v4_compress", "v4_indexer_prep",
           "v4_indexer_topk", "v4_sparse_mqa_fwd", "v4_grouped_o_proj", "v4_attn_layer_fwd",
           "v4_last_error", "v4_get_device_status", "v4_reset_device_status", "v4_launch_count",
           "v4_profile_enable", "v4_profile_count", "v4_profile_get", "v4_sparse_mqa_fwd_noalloc",
           "v4_bwd_workspace_size", "v4_sparse_mqa_bwd", "v4_quantize_e4m3", "v4_indexer_topk_e4m3",
           "v4_q_proj", "v4_indexer_kl_target", "v4_selftest_wait_timeout", "v4_build_info"]
PROFILE_KINDS = {0: "compress", 1: "window_rotate", 2: "indexer_prep", 3: "indexer_scores", 4: "topk",
                 5: "attention", 6: "o_proj", 7: "bwd_prep", 8: "bwd_attention", 9: "bwd_derotate",
                 10: "indexer_quant", 11: "q_proj", 12: "kl_target"}


class V4Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), msg))
        self.status = status


class v4_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "batch", "seqlen", "n_heads", "head_dim", "rope_dim", "ratio", "overlap", "window", "topk",
        "idx_heads", "idx_dim", "o_groups", "o_rank")] + [
        ("softmax_scale", C.c_float), ("rms_eps", C.c_float), ("dtype", C.c_int32), ("path", C.c_int32),
        ("indexer_fp8", C.c_int32), ("q_begin", C.c_int32)]


class v4_layer_inputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "q", "kv", "ckv", "cscore", "ape", "norm_w", "ickv", "icscore", "iape", "inorm_w", "iq", "w",
        "sink", "inv_freq", "wo_a")]


class v4_layer_outputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("o", "lse", "ent", "ikey", "idx", "iscore", "y")]


_lib = None


def lib(path=None):
    """Load the library (once).  Raises if it has not been built.  The
    environment variable V4ATTN_LIB names another build of it (e.g. the
    bound-checking one, build.DEBUG_LIB)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("V4ATTN_LIB") or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("CUDA library %s is missing: build it with "
                           "sparse_compressed_attention_gb300.build.build()" % path)
    L = C.CDLL(path)
    vp, i32, f32, sz = C.c_void_p, C.c_int32, C.c_float, C.c_size_t
    cfgp = C.POINTER(v4_config)
    sig = {
        "v4_rope_inv_freq": [f32, i32, f32, i32, f32, f32, vp],
        "v4_workspace_size": [cfgp, C.POINTER(sz)],
        "v4_compress": [cfgp, vp, vp, vp, vp, vp, i32, i32, vp, vp],
        "v4_indexer_prep": [cfgp, vp, vp, vp, vp],
        "v4_indexer_topk": [cfgp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp],
        "v4_quantize_e4m3": [vp, C.c_int64, i32, vp, vp, vp],
        "v4_indexer_topk_e4m3": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "v4_sparse_mqa_fwd": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "v4_sparse_mqa_fwd_noalloc": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
        "v4_grouped_o_proj": [cfgp, vp, vp, vp, vp],
        "v4_q_proj": [cfgp, vp, i32, vp, i32, vp, vp, vp, vp, vp],
        "v4_indexer_kl_target": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "v4_bwd_workspace_size": [cfgp, C.POINTER(sz)],
        "v4_sparse_mqa_bwd": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "v4_attn_layer_fwd": [cfgp, C.POINTER(v4_layer_inputs), C.POINTER(v4_layer_outputs), vp, sz, vp],
        "v4_get_device_status": [vp, C.POINTER(i32)],
        "v4_reset_device_status": [vp],
        "v4_profile_enable": [i32],
        "v4_profile_get": [i32, C.POINTER(i32), C.POINTER(f32)],
        "v4_selftest_wait_timeout": [i32, vp],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_int
    L.v4_last_error.argtypes = []
    L.v4_last_error.restype = C.c_char_p
    L.v4_build_info.argtypes = []
    L.v4_build_info.restype = C.c_char_p
    L.v4_launch_count.argtypes = []
    L.v4_launch_count.restype = C.c_uint64
    L.v4_profile_count.argtypes = []
    L.v4_profile_count.restype = C.c_int32
    _lib = L
    return L


def _check(status):
    if status != V4_OK:
        raise V4Error(status, lib().v4_last_error().decode())


def make_config(B, S, H, D, R, ratio=0, overlap=0, window=128, topk=0, Hi=64, Di=128,
                o_groups=8, o_rank=1024, scale=0.0, eps=1e-6, dtype="bf16", path=V4_PATH_AUTO,
                indexer_fp8=0, q_begin=0):
    """v4_config; q_begin > 0 restricts the call to query positions q_begin..S-1
    (row tensors then hold S - q_begin rows per sequence)."""
    return v4_config(B, S, H, D, R, ratio, overlap, window, topk, Hi, Di, o_groups, o_rank,
                     scale, eps, V4_BF16 if dtype == "bf16" else V4_F32, path, int(indexer_fp8), int(q_begin))


def config_from_preset(p, **over):
    q = dict(p)
    q.update(over)
    return make_config(q["B"], q["S"], q["H"], q["D"], q["R"], q["ratio"], q["overlap"], q["W"],
                       q["K"], q["Hi"], q["Di"], dtype=q["dtype"], path=q.get("path", V4_PATH_AUTO),
                       eps=q.get("eps", 1e-6), scale=q.get("scale", 0.0),
                       indexer_fp8=q.get("indexer_fp8", 0), q_begin=q.get("q_begin", 0))


def _storage(cfg):
    return torch.bfloat16 if cfg.dtype == V4_BF16 else torch.float32


def _ptr(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def v4_rope_inv_freq(theta, rope_dim, yarn_factor=1.0, original_len=0, beta_fast=32.0, beta_slow=1.0):
    """Host-built inverse-frequency table (float32 CPU tensor of rope_dim/2)."""
    out = (C.c_float * (rope_dim // 2))()
    _check(lib().v4_rope_inv_freq(theta, rope_dim, yarn_factor, original_len, beta_fast, beta_slow, out))
    return torch.tensor(list(out), dtype=torch.float32)


def v4_workspace_size(cfg):
    n = C.c_size_t(0)
    _check(lib().v4_workspace_size(C.byref(cfg), C.byref(n)))
    return n.value


def alloc_workspace(cfg, device=None):
    return torch.empty(max(v4_workspace_size(cfg), 256), dtype=torch.uint8, device=device or "cuda")


def v4_compress(cfg, ckv, cscore, ape, norm_w, inv_freq, dim, hadamard, out, stream=None):
    dt = _storage(cfg)
    _check(lib().v4_compress(C.byref(cfg), _ptr(ckv, "ckv", dt), _ptr(cscore, "cscore", dt),
                             _ptr(ape, "ape", torch.float32),
                             _ptr(norm_w, "norm_w", torch.float32, optional=True),
                             _ptr(inv_freq, "inv_freq", torch.float32, optional=cfg.rope_dim == 0), int(dim), int(hadamard),
                             _ptr(out, "out", dt, optional=out is None), _stream(stream)))
    return out


def v4_indexer_prep(cfg, iq, inv_freq, iq_prep, stream=None):
    dt = _storage(cfg)
    _check(lib().v4_indexer_prep(C.byref(cfg), _ptr(iq, "iq", dt), _ptr(inv_freq, "inv_freq", torch.float32, optional=cfg.rope_dim == 0),
                                 _ptr(iq_prep, "iq_prep", dt), _stream(stream)))
    return iq_prep


def v4_indexer_topk(cfg, iq, iq_prepared, ikey, w, inv_freq, idx, iscore, workspace, stream=None):
    dt = _storage(cfg)
    _check(lib().v4_indexer_topk(C.byref(cfg), _ptr(iq, "iq", dt), int(iq_prepared),
                                 _ptr(ikey, "ikey", dt, optional=True), _ptr(w, "w", torch.float32),
                                 _ptr(inv_freq, "inv_freq", torch.float32, optional=True),
                                 _ptr(idx, "idx", torch.int32),
                                 _ptr(iscore, "iscore", torch.float32, optional=True),
                                 _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                 _stream(stream)))
    return idx


def v4_quantize_e4m3(x, codes, scales, stream=None):
    """x [..., dim] bf16 -> codes [..., dim] uint8 (E4M3 bytes), scales [...] fp32."""
    dim = x.shape[-1]
    rows = x.numel() // dim if dim else 0
    _check(lib().v4_quantize_e4m3(_ptr(x, "x", torch.bfloat16), rows, dim, _ptr(codes, "codes", torch.uint8),
                                  _ptr(scales, "scales", torch.float32), _stream(stream)))
    return codes, scales


def v4_indexer_topk_e4m3(cfg, q_codes, q_scales, k_codes, k_scales, w, idx, iscore, workspace, stream=None):
    _check(lib().v4_indexer_topk_e4m3(C.byref(cfg), _ptr(q_codes, "q_codes", torch.uint8),
                                      _ptr(q_scales, "q_scales", torch.float32),
                                      _ptr(k_codes, "k_codes", torch.uint8, optional=True),
                                      _ptr(k_scales, "k_scales", torch.float32, optional=True),
                                      _ptr(w, "w", torch.float32), _ptr(idx, "idx", torch.int32),
                                      _ptr(iscore, "iscore", torch.float32, optional=True),
                                      _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                      _stream(stream)))
    return idx


def v4_sparse_mqa_fwd(cfg, q, kv, ent, idx, sink, inv_freq, o, lse, workspace, stream=None):
    dt = _storage(cfg)
    _check(lib().v4_sparse_mqa_fwd(C.byref(cfg), _ptr(q, "q", dt), _ptr(kv, "kv", dt),
                                   _ptr(ent, "ent", dt, optional=True),
                                   _ptr(idx, "idx", torch.int32, optional=True),
                                   _ptr(sink, "sink", torch.float32, optional=True),
                                   _ptr(inv_freq, "inv_freq", torch.float32, optional=cfg.rope_dim == 0),
                                   _ptr(o, "o", dt), _ptr(lse, "lse", torch.float32, optional=True),
                                   _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                   _stream(stream)))
    return o


def v4_sparse_mqa_fwd_noalloc(cfg, q, kv, ent, idx, sink, inv_freq, o, lse, stream=None):
    """v4_sparse_mqa_fwd with library-owned scratch (no workspace argument)."""
    dt = _storage(cfg)
    _check(lib().v4_sparse_mqa_fwd_noalloc(C.byref(cfg), _ptr(q, "q", dt), _ptr(kv, "kv", dt),
                                           _ptr(ent, "ent", dt, optional=True),
                                           _ptr(idx, "idx", torch.int32, optional=True),
                                           _ptr(sink, "sink", torch.float32, optional=True),
                                           _ptr(inv_freq, "inv_freq", torch.float32, optional=cfg.rope_dim == 0),
                                           _ptr(o, "o", dt), _ptr(lse, "lse", torch.float32, optional=True),
                                           _stream(stream)))
    return o


def v4_bwd_workspace_size(cfg):
    n = C.c_size_t(0)
    _check(lib().v4_bwd_workspace_size(C.byref(cfg), C.byref(n)))
    return n.value


def alloc_bwd_workspace(cfg, device=None):
    return torch.empty(max(v4_bwd_workspace_size(cfg), 256), dtype=torch.uint8, device=device or "cuda")


def v4_sparse_mqa_bwd(cfg, q, kv, ent, idx, sink, inv_freq, o, lse, dout, dq, dkv, dent, dsink, workspace,
                      stream=None):
    """Gradients of sum(dout * o) for v4_sparse_mqa_fwd; dq, dkv, dent, dsink are written."""
    dt = _storage(cfg)
    _check(lib().v4_sparse_mqa_bwd(C.byref(cfg), _ptr(q, "q", dt), _ptr(kv, "kv", dt),
                                   _ptr(ent, "ent", dt, optional=True),
                                   _ptr(idx, "idx", torch.int32, optional=True),
                                   _ptr(sink, "sink", torch.float32, optional=True),
                                   _ptr(inv_freq, "inv_freq", torch.float32),
                                   _ptr(o, "o", dt), _ptr(lse, "lse", torch.float32), _ptr(dout, "dout", dt),
                                   _ptr(dq, "dq", dt), _ptr(dkv, "dkv", torch.float32),
                                   _ptr(dent, "dent", torch.float32, optional=True),
                                   _ptr(dsink, "dsink", torch.float32, optional=True),
                                   _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                   _stream(stream)))
    return dq, dkv, dent, dsink


def v4_q_proj(cfg, qlat, wq, q, q_norm=1, q_norm_w=None, wiq=None, iq=None, stream=None):
    """q = (per-head RMSNorm of) qlat @ wq, and iq = qlat @ wiq when wiq is given."""
    _check(lib().v4_q_proj(C.byref(cfg), _ptr(qlat, "qlat", torch.bfloat16), int(qlat.shape[-1]),
                           _ptr(wq, "wq", torch.bfloat16), int(q_norm),
                           _ptr(q_norm_w, "q_norm_w", torch.float32, optional=True),
                           _ptr(wiq, "wiq", torch.bfloat16, optional=True), _ptr(q, "q", torch.bfloat16),
                           _ptr(iq, "iq", torch.bfloat16, optional=True), _stream(stream)))
    return q, iq


def v4_indexer_kl_target(cfg, q, ent, idx, lse, iscore, inv_freq, target, loss, dscore, workspace, stream=None):
    """Distillation target of the indexer (and, with iscore, the KL loss and its gradient)."""
    dt = _storage(cfg)
    _check(lib().v4_indexer_kl_target(C.byref(cfg), _ptr(q, "q", dt), _ptr(ent, "ent", dt, optional=True),
                                      _ptr(idx, "idx", torch.int32), _ptr(lse, "lse", torch.float32),
                                      _ptr(iscore, "iscore", torch.float32, optional=True),
                                      _ptr(inv_freq, "inv_freq", torch.float32, optional=True),
                                      _ptr(target, "target", torch.float32),
                                      _ptr(loss, "loss", torch.float32, optional=True),
                                      _ptr(dscore, "dscore", torch.float32, optional=True),
                                      _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))
    return target


def v4_grouped_o_proj(cfg, o, wo_a, y, stream=None):
    dt = _storage(cfg)
    _check(lib().v4_grouped_o_proj(C.byref(cfg), _ptr(o, "o", dt), _ptr(wo_a, "wo_a", dt),
                                   _ptr(y, "y", dt), _stream(stream)))
    return y


_IN_F32 = {"ape", "norm_w", "iape", "inorm_w", "w", "sink", "inv_freq"}


def v4_attn_layer_fwd(cfg, inputs, outputs, workspace, stream=None):
    """inputs / outputs: dicts keyed like v4_layer_inputs / v4_layer_outputs."""
    dt = _storage(cfg)
    vin = v4_layer_inputs()
    for name, _ in v4_layer_inputs._fields_:
        t = inputs.get(name)
        setattr(vin, name, _ptr(t, name, torch.float32 if name in _IN_F32 else dt, optional=True))
    vout = v4_layer_outputs()
    odt = {"lse": torch.float32, "iscore": torch.float32, "idx": torch.int32}
    for name, _ in v4_layer_outputs._fields_:
        t = outputs.get(name)
        setattr(vout, name, _ptr(t, name, odt.get(name, dt), optional=True))
    _check(lib().v4_attn_layer_fwd(C.byref(cfg), C.byref(vin), C.byref(vout),
                                   _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                   _stream(stream)))
    return outputs


def v4_last_error():
    return lib().v4_last_error().decode()


def v4_build_info():
    return lib().v4_build_info().decode()


def v4_get_device_status(stream=None):
    v = C.c_int32(0)
    _check(lib().v4_get_device_status(_stream(stream), C.byref(v)))
    return v.value


def v4_reset_device_status(stream=None):
    _check(lib().v4_reset_device_status(_stream(stream)))


def v4_selftest_wait_timeout(limit_us, stream=None):
    """Launch the self-test kernel whose bounded wait runs out (see the header)."""
    _check(lib().v4_selftest_wait_timeout(int(limit_us), _stream(stream)))


def v4_launch_count():
    return int(lib().v4_launch_count())


def v4_profile_enable(on=True):
    _check(lib().v4_profile_enable(1 if on else 0))


def v4_profile_count():
    return int(lib().v4_profile_count())


def v4_profile_get(i):
    """(kind name, milliseconds) of launch record i."""
    k, ms = C.c_int32(0), C.c_float(0.0)
    _check(lib().v4_profile_get(int(i), C.byref(k), C.byref(ms)))
    return PROFILE_KINDS.get(k.value, str(k.value)), float(ms.value)


def v4_profile_records():
    return [v4_profile_get(i) for i in range(v4_profile_count())]
