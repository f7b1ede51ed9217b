"""GB300 (sm_103a) Kimi Delta Attention operator.

The compute lives in ``libkda.so`` (hand-written CUDA kernels behind the C ABI
declared in ``include/kda.h``).  This module is the thin Python binding: it
turns torch tensors into pointers and sizes, calls the C entry points of the
same names and raises on a non-OK status.  It performs no arithmetic of the
method and has no fallback: if the library is missing, every call raises.

    kda_prefill(q, k, v, g, beta, ...)  chunk-parallel prefill, packed batch
    kda_prefill_noalloc(...)            the same, allocating nothing (fixed scratch array)
    kda_prefill_checkpointed(...)       the same, plus state checkpoints every `interval` tokens
    kda_prefill_gated(q, k, v, z, a_log, beta_logit, ...)   the same, from gate logits
    kda_prefill_output_gated(q, k, v, g, beta, gate_logit, ...)   the same, then the output gate
    kda_prefill_scalar_decay(q, k, v, g_head, beta, ...)   Gated DeltaNet / the delta rule
    kda_backward(q, k, v, g, beta, d_out, ...)   gradients of kda_prefill
    kda_output_gate(out, gate_logit, ...)   the output gate alone, in place
    kda_qkv_prologue(x_q, x_k, x_v, conv_weight, ...)   ShortConv, Swish, L2Norm -> q, k, v
    kda_decode(q, k, v, g, beta, state) one-token in-place state update
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["KdaError", "kda_prefill", "kda_prefill_noalloc", "kda_prefill_checkpointed", "kda_prefill_gated",
           "kda_prefill_output_gated", "kda_prefill_scalar_decay", "kda_backward",
           "kda_output_gate", "kda_qkv_prologue", "checkpoint_count", "kda_decode",
           "kda_status_string", "lib", "library_path",
           "kda_get_last_device_error", "kda_selftest_timeout",
           "PREFILL_DEFAULT", "PREFILL_FP32", "PREFILL_TC", "PREFILL_TC_SPLIT", "PREFILL_TC_2PASS", "Dims"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK = 0
DTYPE_F32, DTYPE_BF16 = 0, 1
PREFILL_DEFAULT, PREFILL_FP32, PREFILL_TC, PREFILL_TC_SPLIT, PREFILL_TC_2PASS = 0, 1, 2, 3, 4
CHUNK = 32   # chunk length of the prefill kernels (KDA_CHUNK)
_DTYPES = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = kda_status_string(status)
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class Dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("variant", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libkda.so (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback")
        L = ctypes.CDLL(_LIB_PATH)
        vp, fp = ctypes.c_void_p, ctypes.c_void_p
        L.kda_prefill.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, fp, vp, vp, fp, vp]
        L.kda_prefill.restype = ctypes.c_int
        L.kda_prefill_noalloc.argtypes = L.kda_prefill.argtypes
        L.kda_prefill_noalloc.restype = ctypes.c_int
        L.kda_prefill_checkpointed.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, fp, vp, vp,
                                               fp, fp, ctypes.c_int64, ctypes.c_int64, vp]
        L.kda_prefill_checkpointed.restype = ctypes.c_int
        L.kda_prefill_gated.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, fp, fp, fp, vp, vp, fp,
                                        vp]
        L.kda_prefill_gated.restype = ctypes.c_int
        L.kda_prefill_output_gated.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, vp, fp,
                                               ctypes.c_float, fp, vp, vp, fp, vp]
        L.kda_prefill_output_gated.restype = ctypes.c_int
        L.kda_prefill_scalar_decay.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, fp, vp, vp,
                                               fp, vp]
        L.kda_prefill_scalar_decay.restype = ctypes.c_int
        L.kda_backward.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, fp, vp, fp,
                                   ctypes.c_int64, vp, fp, vp, vp, vp, fp, fp, fp, vp]
        L.kda_backward.restype = ctypes.c_int
        L.kda_output_gate.argtypes = [ctypes.POINTER(Dims), vp, vp, fp, ctypes.c_float, vp]
        L.kda_output_gate.restype = ctypes.c_int
        L.kda_qkv_prologue.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, vp, vp, vp,
                                       vp, fp, ctypes.c_float, vp]
        L.kda_qkv_prologue.restype = ctypes.c_int
        L.kda_decode.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, fp, fp, fp, vp, vp]
        L.kda_decode.restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_last_cuda_error.restype = ctypes.c_char_p
        L.kda_version.restype = ctypes.c_int32
        L.kda_get_last_device_error.argtypes = [vp]
        L.kda_get_last_device_error.restype = ctypes.c_int
        L.kda_selftest_timeout.argtypes = [vp]
        L.kda_selftest_timeout.restype = ctypes.c_int
        _lib = L
    return _lib


def kda_get_last_device_error(stream=None) -> int:
    """Synchronise `stream` and return (then clear) the device status: 0 or
    4 (KDA_ERR_TIMEOUT) if a bounded device-side wait gave up."""
    return int(lib().kda_get_last_device_error(_stream(stream)))


def kda_selftest_timeout(stream=None) -> None:
    """Enqueue the diagnostic kernel whose bounded wait is made to give up."""
    _check(lib().kda_selftest_timeout(_stream(stream)), "kda_selftest_timeout")


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, where: str):
    if st != KDA_OK:
        detail = lib().kda_last_cuda_error().decode() if st == 3 else ""
        raise KdaError(st, where, detail)


def _require(t, name, dtype=None, ndim=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def _prefill_args(q, k, v, g, beta, init_state, cu_seqlens, num_seqs, out, final_state,
                  out_dtype, variant, return_final_state):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, ndim=3)
    _require(g, "g", torch.float32, 3)   # None: the gated call, which has no g
    _require(beta, "beta", torch.float32, 2)
    _require(init_state, "init_state", torch.float32, 4)
    _require(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, fp32 or bf16")
    T, H, dk = q.shape
    dv = v.shape[2]
    if (k.shape != q.shape or (g is not None and g.shape != q.shape) or v.shape[:2] != (T, H)
            or beta.shape != (T, H)):
        raise ValueError("inconsistent q/k/v/g/beta shapes")
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
    else:
        N = 1 if num_seqs is None else int(num_seqs)
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((T, H, dv), dtype=out_dtype, device=q.device)
    _require(out, "out", out_dtype, 3)
    if final_state is None and return_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    _require(final_state, "final_state", torch.float32, 4)
    dims = Dims(N, T, H, dk, dv, _DTYPES[q.dtype], _DTYPES[out_dtype], int(variant))
    return dims, out, final_state


def checkpoint_count(total_tokens, interval, cu_seqlens=None, num_seqs=1):
    """Rows kda_prefill_checkpointed writes: sum over sequences of
    floor(length / interval) (cu_seqlens is copied to the host to count)."""
    if cu_seqlens is not None:
        cu = cu_seqlens.detach().to("cpu").tolist()
        return sum(max(0, b - a) // interval for a, b in zip(cu[:-1], cu[1:]))
    return int(num_seqs) * ((total_tokens // max(1, int(num_seqs))) // interval)


def kda_prefill_checkpointed(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, interval,
                             num_seqs=None, checkpoints=None, out=None, final_state=None,
                             out_dtype=None, variant=PREFILL_DEFAULT, return_final_state=True,
                             stream=None):
    """Prefill that also writes the state after every `interval` tokens of each
    sequence (C entry point ``kda_prefill_checkpointed``).  Returns
    ``(out, final_state, checkpoints)``; checkpoints [rows, H, d_k, d_v] fp32,
    sequence by sequence (see include/kda.h)."""
    dims, out, final_state = _prefill_args(q, k, v, g, beta, init_state, cu_seqlens, num_seqs,
                                           out, final_state, out_dtype, variant,
                                           return_final_state)
    if checkpoints is None:
        rows = checkpoint_count(q.shape[0], int(interval), cu_seqlens, dims.num_seqs)
        checkpoints = torch.empty((rows, q.shape[1], q.shape[2], v.shape[2]),
                                  dtype=torch.float32, device=q.device)
    _require(checkpoints, "checkpoints", torch.float32, 4)
    st = lib().kda_prefill_checkpointed(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                                        _ptr(out), _ptr(final_state),
                                        _ptr(checkpoints) if checkpoints.numel() else None,
                                        int(interval), int(checkpoints.shape[0]), _stream(stream))
    _check(st, "kda_prefill_checkpointed")
    return out, final_state, checkpoints


def kda_prefill_gated(q, k, v, z, a_log, beta_logit, init_state=None, cu_seqlens=None, *,
                      num_seqs=None, out=None, final_state=None, out_dtype=None,
                      variant=PREFILL_DEFAULT, return_final_state=True, stream=None):
    """Prefill with the gate prologue fused in (C entry point
    ``kda_prefill_gated``): g = -5 Sigmoid(e^{a_log[h]} z) and beta =
    Sigmoid(beta_logit) are formed inside the kernel.  z has the dtype and
    shape of k; a_log fp32 [H]; beta_logit fp32 [T, H].  Returns
    ``(out, final_state)``."""
    if z.dtype != k.dtype or z.shape != k.shape:
        raise ValueError("z must have the dtype and shape of k")
    _require(z, "z", k.dtype, 3)
    _require(a_log, "a_log", torch.float32, 1)
    if a_log.shape[0] != q.shape[1]:
        raise ValueError("a_log must hold one value per head")
    dims, out, final_state = _prefill_args(q, k, v, None, beta_logit, init_state, cu_seqlens,
                                           num_seqs, out, final_state, out_dtype, variant,
                                           return_final_state)
    st = lib().kda_prefill_gated(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                                 _ptr(a_log), _ptr(beta_logit), _ptr(init_state),
                                 _ptr(cu_seqlens), _ptr(out), _ptr(final_state), _stream(stream))
    _check(st, "kda_prefill_gated")
    return out, final_state


def kda_prefill_output_gated(q, k, v, g, beta, gate_logit, norm_weight=None, eps=1e-6,
                             init_state=None, cu_seqlens=None, *, num_seqs=None, out=None,
                             final_state=None, out_dtype=None, variant=PREFILL_DEFAULT,
                             return_final_state=True, stream=None):
    """Prefill followed by the output gate (C entry point
    ``kda_prefill_output_gated``): out = Sigmoid(gate_logit) * o~ /
    sqrt(mean over d_v of o~^2 + eps) * norm_weight, per token and head.
    gate_logit has the dtype and shape of v; norm_weight fp32 [d_v] or None.
    Returns ``(out, final_state)``."""
    if gate_logit.dtype != v.dtype or gate_logit.shape != v.shape:
        raise ValueError("gate_logit must have the dtype and shape of v")
    _require(gate_logit, "gate_logit", v.dtype, 3)
    _require(norm_weight, "norm_weight", torch.float32, 1)
    if norm_weight is not None and norm_weight.shape[0] != v.shape[2]:
        raise ValueError("norm_weight must hold one value per value channel")
    dims, out, final_state = _prefill_args(q, k, v, g, beta, init_state, cu_seqlens, num_seqs,
                                           out, final_state, out_dtype, variant,
                                           return_final_state)
    st = lib().kda_prefill_output_gated(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(gate_logit), _ptr(norm_weight),
                                        ctypes.c_float(eps), _ptr(init_state), _ptr(cu_seqlens),
                                        _ptr(out), _ptr(final_state), _stream(stream))
    _check(st, "kda_prefill_output_gated")
    return out, final_state


def kda_prefill_scalar_decay(q, k, v, g_head, beta, init_state=None, cu_seqlens=None, *,
                             num_seqs=None, out=None, final_state=None, out_dtype=None,
                             variant=PREFILL_DEFAULT, return_final_state=True, stream=None):
    """Gated DeltaNet prefill, one log-decay per (token, head): g_head fp32
    [T, H]; or the delta rule with g_head None (C entry point
    ``kda_prefill_scalar_decay``).  Returns ``(out, final_state)``."""
    _require(g_head, "g_head", torch.float32, 2)
    if g_head is not None and g_head.shape != q.shape[:2]:
        raise ValueError("g_head must be [T, H]")
    dims, out, final_state = _prefill_args(q, k, v, None, beta, init_state, cu_seqlens, num_seqs,
                                           out, final_state, out_dtype, variant,
                                           return_final_state)
    st = lib().kda_prefill_scalar_decay(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(g_head), _ptr(beta), _ptr(init_state),
                                        _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                        _stream(stream))
    _check(st, "kda_prefill_scalar_decay")
    return out, final_state


def kda_backward(q, k, v, g, beta, d_out, d_final_state=None, init_state=None, cu_seqlens=None,
                 *, chunk_states=None, num_seqs=None, grad_dtype=None, stream=None):
    """Gradients of kda_prefill (C entry point ``kda_backward``) for the
    upstream gradients d_out [T, H, d_v] (dtype of q) and d_final_state
    [N, H, d_k, d_v] fp32 (None: zero).  ``chunk_states`` are the forward's
    states at every chunk start, as kda_prefill_checkpointed writes them with
    interval CHUNK; when None they are computed here by that call.  Returns a
    dict with dq, dk, dv (``grad_dtype``, default the dtype of q), dg, dbeta
    and d_init_state (fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_out, "d_out")):
        _require(t, n, q.dtype, 3)
    _require(g, "g", torch.float32, 3)
    _require(beta, "beta", torch.float32, 2)
    _require(init_state, "init_state", torch.float32, 4)
    _require(d_final_state, "d_final_state", torch.float32, 4)
    _require(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if q.dtype not in _DTYPES:
        raise ValueError("q, k, v must be fp32 or bf16")
    T, H, dk = q.shape
    dv = v.shape[2]
    if d_out.shape != v.shape:
        raise ValueError("d_out must have the shape of v")
    N = cu_seqlens.shape[0] - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    if chunk_states is None:
        _, _, chunk_states = kda_prefill_checkpointed(q, k, v, g, beta, init_state, cu_seqlens,
                                                      interval=CHUNK, num_seqs=N,
                                                      return_final_state=False, stream=stream)
    _require(chunk_states, "chunk_states", torch.float32, 4)
    grad_dtype = grad_dtype or q.dtype
    dev = q.device
    res = dict(dq=torch.empty((T, H, dk), dtype=grad_dtype, device=dev),
               dk=torch.empty((T, H, dk), dtype=grad_dtype, device=dev),
               dv=torch.empty((T, H, dv), dtype=grad_dtype, device=dev),
               dg=torch.empty((T, H, dk), dtype=torch.float32, device=dev),
               dbeta=torch.empty((T, H), dtype=torch.float32, device=dev),
               d_init_state=torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev))
    dims = Dims(N, T, H, dk, dv, _DTYPES[q.dtype], _DTYPES[grad_dtype], 0)
    cs = chunk_states if chunk_states.numel() else None
    st = lib().kda_backward(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            _ptr(init_state), _ptr(cu_seqlens), _ptr(cs),
                            int(chunk_states.shape[0]) if cs is not None else 0, _ptr(d_out),
                            _ptr(d_final_state), _ptr(res["dq"]), _ptr(res["dk"]),
                            _ptr(res["dv"]), _ptr(res["dg"]), _ptr(res["dbeta"]),
                            _ptr(res["d_init_state"]), _stream(stream))
    _check(st, "kda_backward")
    return res


def kda_output_gate(out, gate_logit, norm_weight=None, eps=1e-6, stream=None):
    """The output gate in place on ``out`` [T, H, d_v] (C entry point
    ``kda_output_gate``): out = Sigmoid(gate_logit) * out / sqrt(mean over d_v
    of out^2 + eps) * norm_weight.  gate_logit [T, H, d_v] fp32 or bf16;
    norm_weight fp32 [d_v] or None.  Returns ``out``."""
    _require(out, "out", ndim=3)
    _require(gate_logit, "gate_logit", ndim=3)
    _require(norm_weight, "norm_weight", torch.float32, 1)
    if out.dtype not in _DTYPES or gate_logit.dtype not in _DTYPES:
        raise ValueError("out and gate_logit must be fp32 or bf16")
    if gate_logit.shape != out.shape:
        raise ValueError("gate_logit must have the shape of out")
    T, H, dv = out.shape
    if norm_weight is not None and norm_weight.shape[0] != dv:
        raise ValueError("norm_weight must hold one value per value channel")
    dims = Dims(1, T, H, dv, dv, _DTYPES[gate_logit.dtype], _DTYPES[out.dtype], 0)
    _check(lib().kda_output_gate(ctypes.byref(dims), _ptr(out), _ptr(gate_logit),
                                 _ptr(norm_weight), ctypes.c_float(eps), _stream(stream)),
           "kda_output_gate")
    return out


def kda_qkv_prologue(x_q, x_k, x_v, conv_weight, cu_seqlens=None, conv_state=None, *,
                     num_seqs=None, eps=1e-6, out_dtype=None, q=None, k=None, v=None,
                     conv_state_out=None, return_conv_state=True, stream=None):
    """q, k, v from their projections (C entry point ``kda_qkv_prologue``):
    per channel the causal width-4 convolution over each sequence, Swish, and
    for q and k the L2 normalisation over the head's d channels.

    x_q, x_k, x_v [T, H, d] fp32 or bf16 (one dtype); conv_weight fp32
    [3, H, d, 4] (streams q, k, v; tap 3 on the current token); cu_seqlens
    int32 [N+1] or None (``num_seqs`` equal sequences, default 1); conv_state
    fp32 [N, 3, 3, H, d] or None (zeros).  Returns ``(q, k, v, conv_state_out)``
    (the last, fp32 [N, 3, 3, H, d], is None unless ``return_conv_state`` or
    a buffer is given)."""
    for t, n in ((x_q, "x_q"), (x_k, "x_k"), (x_v, "x_v")):
        _require(t, n, ndim=3)
    _require(conv_weight, "conv_weight", torch.float32, 4)
    _require(conv_state, "conv_state", torch.float32, 5)
    _require(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if x_q.dtype not in _DTYPES or x_k.dtype != x_q.dtype or x_v.dtype != x_q.dtype:
        raise ValueError("x_q, x_k, x_v must share one dtype, fp32 or bf16")
    if x_k.shape != x_q.shape or x_v.shape != x_q.shape:
        raise ValueError("x_q, x_k, x_v must have one shape [T, H, d]")
    T, H, d = x_q.shape
    if conv_weight.shape != (3, H, d, 4):
        raise ValueError("conv_weight must be [3, H, d, 4]")
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
    else:
        N = 1 if num_seqs is None else int(num_seqs)
    if conv_state is not None and conv_state.shape != (N, 3, 3, H, d):
        raise ValueError("conv_state must be [N, 3, 3, H, d]")
    odt = x_q.dtype if out_dtype is None else out_dtype
    if odt not in _DTYPES:
        raise ValueError("out_dtype must be fp32 or bf16")
    outs = []
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t is None:
            t = torch.empty((T, H, d), dtype=odt, device=x_q.device)
        _require(t, n, odt, 3)
        if t.shape != (T, H, d):
            raise ValueError(f"{n} must be [T, H, d]")
        outs.append(t)
    if conv_state_out is None and return_conv_state:
        conv_state_out = torch.empty((N, 3, 3, H, d), dtype=torch.float32, device=x_q.device)
    _require(conv_state_out, "conv_state_out", torch.float32, 5)
    if conv_state_out is not None and conv_state_out.shape != (N, 3, 3, H, d):
        raise ValueError("conv_state_out must be [N, 3, 3, H, d]")
    dims = Dims(N, T, H, d, d, _DTYPES[x_q.dtype], _DTYPES[odt], 0)
    _check(lib().kda_qkv_prologue(ctypes.byref(dims), _ptr(x_q), _ptr(x_k), _ptr(x_v),
                                  _ptr(conv_weight), _ptr(conv_state), _ptr(cu_seqlens),
                                  _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
                                  _ptr(conv_state_out), ctypes.c_float(eps), _stream(stream)),
           "kda_qkv_prologue")
    return outs[0], outs[1], outs[2], conv_state_out


def kda_prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, num_seqs=None,
                out=None, final_state=None, out_dtype=None, variant=PREFILL_DEFAULT,
                return_final_state=True, stream=None):
    """Chunked KDA prefill (C entry point ``kda_prefill``).

    q, k [T, H, d_k] and v [T, H, d_v] in fp32 or bf16; g [T, H, d_k] fp32;
    beta [T, H] fp32; init_state [N, H, d_k, d_v] fp32 or None; cu_seqlens
    int32 [N+1] (device) or None (``num_seqs`` equal-length sequences,
    default 1).  Returns ``(out, final_state)``.
    """
    dims, out, final_state = _prefill_args(q, k, v, g, beta, init_state, cu_seqlens, num_seqs,
                                           out, final_state, out_dtype, variant,
                                           return_final_state)
    st = lib().kda_prefill(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                           _stream(stream))
    _check(st, "kda_prefill")
    return out, final_state


def kda_prefill_noalloc(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, num_seqs=None,
                        out=None, final_state=None, out_dtype=None, return_final_state=True,
                        stream=None):
    """kda_prefill through the C entry point ``kda_prefill_noalloc``: the split
    kernel on the library's fixed scratch array, for callers that may not
    allocate device memory during a call.  The library allocates nothing; pass
    ``out`` (and ``final_state``) to allocate nothing here either.  Calls that
    overlap on the GPU share the array and must be serialised."""
    dims, out, final_state = _prefill_args(q, k, v, g, beta, init_state, cu_seqlens, num_seqs,
                                           out, final_state, out_dtype, PREFILL_TC_SPLIT,
                                           return_final_state)
    st = lib().kda_prefill_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
                                   _ptr(final_state), _stream(stream))
    _check(st, "kda_prefill_noalloc")
    return out, final_state


def kda_decode(q, k, v, g, beta, state, *, out=None, out_dtype=None, stream=None):
    """One decode step (C entry point ``kda_decode``): q, k, g [N, H, d_k];
    v [N, H, d_v]; beta [N, H]; state [N, H, d_k, d_v] fp32, updated in place.
    Returns ``out`` [N, H, d_v]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, ndim=3)
    _require(g, "g", torch.float32, 3)
    _require(beta, "beta", torch.float32, 2)
    _require(state, "state", torch.float32, 4)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, fp32 or bf16")
    N, H, dk = q.shape
    dv = v.shape[2]
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((N, H, dv), dtype=out_dtype, device=q.device)
    _require(out, "out", out_dtype, 3)
    dims = Dims(N, N, H, dk, dv, _DTYPES[q.dtype], _DTYPES[out_dtype], 0)
    st = lib().kda_decode(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                          _ptr(state), _ptr(out), _stream(stream))
    _check(st, "kda_decode")
    return out
