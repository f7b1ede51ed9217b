"""fp64 CPU oracle of the Kimi Delta Attention recurrence.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The CUDA product path
never imports this package, and this package imports nothing from it.

The arithmetic lives in ``kda_oracle.c`` (plain C, one token at a time, fp64),
which follows the state-update, delta-form and readout equations of
"Understanding Kimi K3's Attention" and the recurrent walk-through in
"Hybrid Attention", section "KDA: don't write the same information twice".
This module only compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lib = None

G_MIN = -5.0


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -march flags: the same code builds on
    x86_64 and aarch64 and gives the same results)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "kda_oracle.h")))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """Bindings to one compiled copy of the oracle (the default build, or a
    copy compiled elsewhere, e.g. by a test that plants a mistake in a
    scratch copy of the source to show that the pins catch it)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i32 = ctypes.c_int32
        lib.kda_oracle_prefill.argtypes = [i32, i32, i32, i32, i32, dp, dp, dp, dp, dp,
                                           dp, ip, dp, dp, i32]
        lib.kda_oracle_prefill.restype = ctypes.c_int
        lib.kda_oracle_prefill_scalar_decay.argtypes = lib.kda_oracle_prefill.argtypes
        lib.kda_oracle_prefill_scalar_decay.restype = ctypes.c_int
        lib.kda_oracle_backward.argtypes = [i32, i32, i32, i32, i32] + [dp] * 6 + [
            ctypes.POINTER(ctypes.c_int32)] + [dp] * 8 + [i32]
        lib.kda_oracle_backward.restype = ctypes.c_int
        lib.kda_oracle_decode.argtypes = [i32, i32, i32, i32, dp, dp, dp, dp, dp, dp, dp, i32]
        lib.kda_oracle_decode.restype = ctypes.c_int
        lib.kda_oracle_num_cpus.restype = ctypes.c_int
        lib.kda_oracle_gate.argtypes = [i32, i32, i32, dp, dp, dp, dp, dp]
        lib.kda_oracle_output_gate.argtypes = [i32, i32, i32, dp, dp, dp, ctypes.c_double, dp]
        lib.kda_oracle_gate.restype = ctypes.c_int
        lib.kda_oracle_qkv_prologue.argtypes = [i32, i32, i32, i32, ip, dp, dp, dp,
                                                ctypes.c_double, dp, dp]
        lib.kda_oracle_qkv_prologue.restype = ctypes.c_int
        self.lib = lib

    def num_cpus(self) -> int:
        return int(self.lib.kda_oracle_num_cpus())

    def prefill(self, q, k, v, g, beta, init_state=None, cu_seqlens=None, num_seqs=None,
                num_threads: int = 0):
        """Token-by-token KDA over a packed batch, in fp64.

        q, k, g: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H]; init_state:
        [N, H, d_k, d_v] or None (zeros); cu_seqlens: int [N+1] or None (then
        ``num_seqs`` equal-length sequences, default 1).
        Returns (out [T, H, d_v], final_state [N, H, d_k, d_v]), both fp64.
        """
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        T, H, dk = q.shape
        dv = v.shape[2]
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
            N = cu.shape[0] - 1
        else:
            cu = None
            N = 1 if num_seqs is None else int(num_seqs)
        init = _f64(init_state)
        out = np.zeros((T, H, dv), np.float64)
        fin = np.zeros((N, H, dk, dv), np.float64)
        rc = self.lib.kda_oracle_prefill(N, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                         _ptr(beta), _ptr(init), _ptr(cu, ctypes.c_int32),
                                         _ptr(out), _ptr(fin), int(num_threads))
        if rc != 0:
            raise ValueError("kda_oracle_prefill rejected its arguments (shapes, "
                             "cu_seqlens, or gates outside g in [-5,0], beta in [0,1])")
        return out, fin

    def prefill_scalar_decay(self, q, k, v, g_head, beta, init_state=None, cu_seqlens=None,
                             num_seqs=None, num_threads: int = 0):
        """Gated DeltaNet: one log-decay per (token, head), g_head [T, H], or
        None for the delta rule (alpha = 1).  Other arguments and the result as
        :meth:`prefill` (C function ``kda_oracle_prefill_scalar_decay``)."""
        q, k, v, gh, beta, init = (_f64(x) for x in (q, k, v, g_head, beta, init_state))
        T, H, dk = q.shape
        dv = v.shape[2]
        assert gh is None or gh.shape == (T, H)
        cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = (cu.shape[0] - 1) if cu is not None else (1 if num_seqs is None else int(num_seqs))
        out = np.zeros((T, H, dv), np.float64)
        fin = np.zeros((N, H, dk, dv), np.float64)
        rc = self.lib.kda_oracle_prefill_scalar_decay(
            N, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(gh), _ptr(beta), _ptr(init),
            _ptr(cu, ctypes.c_int32), _ptr(out), _ptr(fin), int(num_threads))
        if rc != 0:
            raise ValueError("kda_oracle_prefill_scalar_decay rejected its arguments")
        return out, fin

    def backward(self, q, k, v, g, beta, d_out, d_final_state=None, init_state=None,
                 cu_seqlens=None, num_seqs=None, num_threads: int = 0):
        """Gradients of (out, final_state) = prefill(...) for the upstream
        gradients d_out [T, H, d_v] and d_final_state [N, H, d_k, d_v] (None:
        zero), in fp64 (C function ``kda_oracle_backward``).  Returns a dict
        with dq, dk, dv, dg, dbeta and d_init_state."""
        q, k, v, g, beta, do, dfin, init = (_f64(x) for x in (q, k, v, g, beta, d_out,
                                                              d_final_state, init_state))
        T, H, dk = q.shape
        dv = v.shape[2]
        cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = (cu.shape[0] - 1) if cu is not None else (1 if num_seqs is None else int(num_seqs))
        res = dict(dq=np.zeros((T, H, dk)), dk=np.zeros((T, H, dk)), dv=np.zeros((T, H, dv)),
                   dg=np.zeros((T, H, dk)), dbeta=np.zeros((T, H)),
                   d_init_state=np.zeros((N, H, dk, dv)))
        rc = self.lib.kda_oracle_backward(
            N, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init),
            _ptr(cu, ctypes.c_int32), _ptr(do), _ptr(dfin), _ptr(res["dq"]), _ptr(res["dk"]),
            _ptr(res["dv"]), _ptr(res["dg"]), _ptr(res["dbeta"]), _ptr(res["d_init_state"]),
            int(num_threads))
        if rc != 0:
            raise ValueError("kda_oracle_backward rejected its arguments")
        return res

    def gate(self, z, a_log, beta_logit):
        """g [T, H, d_k] and beta [T, H] (fp64) from the decay logits z
        [T, H, d_k], the per-head log-scales a_log [H] and the beta logits
        [T, H] (C function ``kda_oracle_gate``)."""
        z, a_log, bl = _f64(z), _f64(a_log), _f64(beta_logit)
        T, H, dk = z.shape
        assert a_log.shape == (H,) and bl.shape == (T, H)
        g = np.empty_like(z)
        beta = np.empty_like(bl)
        self.lib.kda_oracle_gate(T, H, dk, _ptr(z), _ptr(a_log), _ptr(bl), _ptr(g), _ptr(beta))
        return g, beta

    def output_gate(self, o, gate_logit, norm_weight=None, eps: float = 1e-6):
        """y = Sigmoid(gate_logit) * RMSNorm(o) * norm_weight over the last axis
        (d_v) of o, gate_logit [T, H, d_v] (fp64); norm_weight [d_v] or None
        (C function ``kda_oracle_output_gate``)."""
        o, gl, w = _f64(o), _f64(gate_logit), _f64(norm_weight)
        T, H, dv = o.shape
        assert gl.shape == o.shape and (w is None or w.shape == (dv,))
        y = np.empty_like(o)
        rc = self.lib.kda_oracle_output_gate(T, H, dv, _ptr(o), _ptr(gl), _ptr(w), float(eps),
                                             _ptr(y))
        if rc != 0:
            raise ValueError("kda_oracle_output_gate rejected its arguments (eps must be > 0)")
        return y

    def qkv_prologue(self, x_q, x_k, x_v, conv_weight, cu_seqlens=None, conv_state=None,
                     eps: float = 1e-6):
        """q, k, v from their projections: per channel the causal width-4
        convolution over each sequence, Swish, and for q and k the L2
        normalisation over the head's d channels (C function
        ``kda_oracle_qkv_prologue``).  x_* [T, H, d]; conv_weight [3, H, d, 4]
        (streams q, k, v; tap 3 on the current token); cu_seqlens int32 [N+1]
        or None (one sequence); conv_state [N, 3, 3, H, d] or None (zeros).
        Returns (q, k, v, conv_state_out), fp64."""
        x = _f64(np.stack([_f64(x_q), _f64(x_k), _f64(x_v)]))
        w = _f64(conv_weight)
        _, T, H, d = x.shape
        cu = (np.array([0, T], np.int32) if cu_seqlens is None
              else np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32)))
        N = cu.shape[0] - 1
        assert w.shape == (3, H, d, 4)
        cs = _f64(conv_state)
        assert cs is None or cs.shape == (N, 3, 3, H, d)
        y = np.empty_like(x)
        cout = np.empty((N, 3, 3, H, d))
        rc = self.lib.kda_oracle_qkv_prologue(N, T, H, d, _ptr(cu, ctypes.c_int32), _ptr(x),
                                              _ptr(w), _ptr(cs), float(eps), _ptr(y), _ptr(cout))
        if rc != 0:
            raise ValueError("kda_oracle_qkv_prologue rejected its arguments")
        return y[0], y[1], y[2], cout

    def decode(self, q, k, v, g, beta, state, num_threads: int = 0, inplace: bool = False):
        """One decode step for N sequences: q, k, g [N, H, d_k]; v [N, H, d_v];
        beta [N, H]; state [N, H, d_k, d_v].  Returns (out, new_state), fp64.
        The input ``state`` is left alone unless ``inplace`` (then it must be
        a C-contiguous float64 array and is updated and returned)."""
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        if inplace:
            if not (isinstance(state, np.ndarray) and state.dtype == np.float64
                    and state.flags.c_contiguous):
                raise ValueError("inplace decode needs a C-contiguous float64 state")
            st = state
        else:
            st = np.array(state, dtype=np.float64, copy=True, order="C")
        N, H, dk = q.shape
        dv = v.shape[2]
        out = np.zeros((N, H, dv), np.float64)
        rc = self.lib.kda_oracle_decode(N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(st), _ptr(out), int(num_threads))
        if rc != 0:
            raise ValueError("kda_oracle_decode rejected its arguments")
        return out, st


def _load() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def num_cpus() -> int:
    return _load().num_cpus()


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def prefill(*args, **kwargs):
    """Module-level form of :meth:`Oracle.prefill` on the default build."""
    return _load().prefill(*args, **kwargs)


def prefill_scalar_decay(*args, **kwargs):
    return _load().prefill_scalar_decay(*args, **kwargs)


def backward(*args, **kwargs):
    return _load().backward(*args, **kwargs)


def gate(*args, **kwargs):
    return _load().gate(*args, **kwargs)


def output_gate(*args, **kwargs):
    return _load().output_gate(*args, **kwargs)


def qkv_prologue(*args, **kwargs):
    return _load().qkv_prologue(*args, **kwargs)


def decode(*args, **kwargs):
    """Module-level form of :meth:`Oracle.decode` on the default build."""
    return _load().decode(*args, **kwargs)
