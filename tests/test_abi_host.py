"""Host-side checks of the C ABI (no GPU needed, no compute launched).

- the library builds and loads, and exports every function include/kda.h declares;
- argument validation rejects bad input with the documented status before
  any launch (every call here is invalid, so nothing reaches the device).
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import Dims, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    _build.build()
    return kda.lib()


def declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "kda_prefill" in names and "kda_decode" in names
    out = subprocess.run(["nm", "-D", "--defined-only", kda.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(kda_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in names:
        assert hasattr(L, n)


def test_status_strings(L):
    for code, name in [(0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARGUMENT"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_CUDA"), (4, "KDA_ERR_TIMEOUT")]:
        assert kda.kda_status_string(code) == name
    assert kda.kda_status_string(99) == "KDA_ERR_UNKNOWN"
    assert L.kda_version() >= 100


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: every call below is rejected
FAKE_MISALIGNED = ctypes.c_void_p(0x10004)


def prefill(L, dims, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, init=None, cu=None,
                out=ctypes.c_void_p(0x20000), fin=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_prefill(d, args["q"], args["k"], args["v"], args["g"], args["beta"],
                         args["init"], args["cu"], args["out"], args["fin"], None)


def decode(L, dims, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=ctypes.c_void_p(0x30000),
                out=ctypes.c_void_p(0x20000))
    args.update(over)
    return L.kda_decode(ctypes.byref(dims), args["q"], args["k"], args["v"], args["g"],
                        args["beta"], args["state"], args["out"], None)


def D(**kw):
    base = dict(num_seqs=1, total_tokens=16, num_heads=2, d_k=128, d_v=128, in_dtype=1,
                out_dtype=1, variant=0)
    base.update(kw)
    return Dims(**base)


@pytest.mark.parametrize("dims,over,want", [
    (None, {}, INVALID),
    (D(num_seqs=-1), {}, INVALID),
    (D(total_tokens=-5), {}, INVALID),
    (D(num_heads=0), {}, INVALID),
    (D(d_k=0), {}, INVALID),
    (D(in_dtype=7), {}, INVALID),
    (D(out_dtype=-1), {}, INVALID),
    (D(variant=9), {}, INVALID),
    (D(d_k=96, d_v=96), {}, UNSUPPORTED),
    (D(d_k=128, d_v=64), {}, UNSUPPORTED),
    (D(d_k=32, d_v=32), {}, UNSUPPORTED),
    (D(), {"q": None}, INVALID),
    (D(), {"g": None}, INVALID),
    (D(), {"beta": None}, INVALID),
    (D(), {"out": None}, INVALID),
    (D(num_seqs=3, total_tokens=16), {}, INVALID),          # T % N != 0 without cu_seqlens
    (D(num_seqs=0, total_tokens=4), {}, INVALID),
    (D(), {"out": FAKE}, INVALID),                           # out aliases q
    (D(num_seqs=2, total_tokens=16), {"init": ctypes.c_void_p(0x40000),
                                       "fin": ctypes.c_void_p(0x40000 + 4096)}, INVALID),
])
def test_prefill_rejects(L, dims, over, want):
    assert prefill(L, dims, **over) == want


def prefill_ckpt(L, dims, interval=64, capacity=2, ckpt=ctypes.c_void_p(0x50000), **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, init=None, cu=None,
                out=ctypes.c_void_p(0x20000), fin=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_prefill_checkpointed(d, args["q"], args["k"], args["v"], args["g"], args["beta"],
                                      args["init"], args["cu"], args["out"], args["fin"], ckpt,
                                      interval, capacity, None)


@pytest.mark.parametrize("kw,want", [
    (dict(interval=0), INVALID),
    (dict(interval=-32), INVALID),
    (dict(interval=48), INVALID),                 # not a multiple of the chunk length
    (dict(interval=1), INVALID),
    (dict(capacity=-1), INVALID),
    (dict(ckpt=None), INVALID),                   # rows requested but no buffer
    (dict(ckpt=ctypes.c_void_p(0x50002)), INVALID),   # misaligned
])
def test_prefill_checkpointed_rejects(L, kw, want):
    assert prefill_ckpt(L, D(), **kw) == want


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(), {"q": None}), (D(num_seqs=3, total_tokens=16), {}),
])
def test_prefill_checkpointed_validates_like_prefill(L, dims, over):
    assert prefill_ckpt(L, dims, **over) == INVALID


def test_prefill_checkpointed_empty_batch_is_ok(L):
    assert prefill_ckpt(L, D(num_seqs=0, total_tokens=0), capacity=0, ckpt=None, q=None, k=None,
                        v=None, g=None, beta=None, out=None) == OK


def prefill_gated(L, dims, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, z=ctypes.c_void_p(0x60000), a=ctypes.c_void_p(0x70000),
                bl=FAKE, init=None, cu=None, out=ctypes.c_void_p(0x20000), fin=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_prefill_gated(d, args["q"], args["k"], args["v"], args["z"], args["a"],
                               args["bl"], args["init"], args["cu"], args["out"], args["fin"],
                               None)


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(), {"z": None}), (D(), {"a": None}),
    (D(), {"bl": None}), (D(), {"q": None}), (D(), {"z": ctypes.c_void_p(0x20000)}),
    (D(num_seqs=3, total_tokens=16), {}),
])
def test_prefill_gated_rejects(L, dims, over):
    assert prefill_gated(L, dims, **over) == INVALID


def test_prefill_gated_empty_batch_is_ok(L):
    assert prefill_gated(L, D(num_seqs=0, total_tokens=0), q=None, k=None, v=None, z=None,
                         a=None, bl=None, out=None) == OK


def prefill_ogated(L, dims, eps=1e-6, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, gl=ctypes.c_void_p(0x60000), w=None,
                init=None, cu=None, out=ctypes.c_void_p(0x20000), fin=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_prefill_output_gated(d, args["q"], args["k"], args["v"], args["g"], args["beta"],
                                      args["gl"], args["w"], ctypes.c_float(eps), args["init"],
                                      args["cu"], args["out"], args["fin"], None)


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(), {"gl": None}), (D(), {"q": None}),
    (D(), {"g": None}), (D(), {"gl": ctypes.c_void_p(0x20000)}),     # gate aliases out
    (D(), {"gl": ctypes.c_void_p(0x60001)}),                         # misaligned bf16 gate
    (D(in_dtype=0), {"gl": ctypes.c_void_p(0x60002)}),               # misaligned fp32 gate
    (D(), {"w": ctypes.c_void_p(0x80002)}),                          # misaligned weight
    (D(), {"eps": 0.0}), (D(), {"eps": -1e-6}), (D(), {"eps": float("nan")}),
    (D(), {"eps": float("inf")}), (D(num_seqs=3, total_tokens=16), {}),
])
def test_prefill_output_gated_rejects(L, dims, over):
    assert prefill_ogated(L, dims, **over) == INVALID


def test_prefill_output_gated_empty_batch_is_ok(L):
    assert prefill_ogated(L, D(num_seqs=0, total_tokens=0), q=None, k=None, v=None, g=None,
                          beta=None, gl=None, out=None) == OK


def prefill_sdecay(L, dims, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, gh=ctypes.c_void_p(0x60000), beta=FAKE, init=None,
                cu=None, out=ctypes.c_void_p(0x20000), fin=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_prefill_scalar_decay(d, args["q"], args["k"], args["v"], args["gh"],
                                      args["beta"], args["init"], args["cu"], args["out"],
                                      args["fin"], None)


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(), {"q": None}), (D(), {"beta": None}),
    (D(), {"out": None}), (D(), {"gh": ctypes.c_void_p(0x60002)}),   # misaligned decay
    (D(num_seqs=3, total_tokens=16), {}), (D(), {"out": FAKE}),
])
def test_prefill_scalar_decay_rejects(L, dims, over):
    assert prefill_sdecay(L, dims, **over) == INVALID


def test_prefill_scalar_decay_empty_batch_is_ok(L):
    assert prefill_sdecay(L, D(num_seqs=0, total_tokens=0), q=None, k=None, v=None, gh=None,
                          beta=None, out=None) == OK


def backward(L, dims, cap=4, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, init=None, cu=None,
                cs=ctypes.c_void_p(0x1000000), do=ctypes.c_void_p(0x98000), dfin=None,
                dq=ctypes.c_void_p(0xa0000), dk=ctypes.c_void_p(0xa8000),
                dv=ctypes.c_void_p(0xb0000), dg=ctypes.c_void_p(0xb8000),
                db=ctypes.c_void_p(0xc0000), dinit=None)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_backward(d, args["q"], args["k"], args["v"], args["g"], args["beta"],
                          args["init"], args["cu"], args["cs"], cap, args["do"], args["dfin"],
                          args["dq"], args["dk"], args["dv"], args["dg"], args["db"],
                          args["dinit"], None)


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(d_k=96, d_v=96), {}), (D(), {"q": None}),
    (D(), {"do": None}), (D(), {"dg": None}), (D(), {"db": None}), (D(), {"dq": None}),
    (D(), {"cap": -1}), (D(total_tokens=64), {"cs": None, "cap": 0}),   # needs chunk states
    (D(), {"cs": ctypes.c_void_p(0x90002)}),                          # misaligned
    (D(), {"dq": FAKE}), (D(), {"dk": ctypes.c_void_p(0x98000)}),     # gradient aliases an input
    (D(num_seqs=3, total_tokens=16), {}),
])
def test_backward_rejects(L, dims, over):
    want = UNSUPPORTED if dims is not None and dims.d_k == 96 else INVALID
    assert backward(L, dims, **over) == want


def test_backward_empty_batch_is_ok(L):
    assert backward(L, D(num_seqs=0, total_tokens=0), cap=0, cs=None, q=None, k=None, v=None,
                    g=None, beta=None, do=None, dq=None, dk=None, dv=None, dg=None,
                    db=None) == OK


@pytest.mark.parametrize("dims,over", [
    (None, {}), (D(num_heads=0), {}), (D(), {"out": None}), (D(), {"gl": None}),
    (D(), {"gl": ctypes.c_void_p(0x20000)}),                    # gate aliases out
    (D(), {"gl": ctypes.c_void_p(0x60001)}), (D(), {"out": ctypes.c_void_p(0x20001)}),
    (D(), {"w": ctypes.c_void_p(0x80002)}), (D(), {"eps": 0.0}), (D(), {"eps": float("nan")}),
])
def test_output_gate_rejects(L, dims, over):
    args = dict(out=ctypes.c_void_p(0x20000), gl=ctypes.c_void_p(0x60000), w=None, eps=1e-6)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    assert L.kda_output_gate(d, args["out"], args["gl"], args["w"], ctypes.c_float(args["eps"]),
                             None) == INVALID


def test_output_gate_no_rows_is_ok(L):
    assert L.kda_output_gate(ctypes.byref(D(total_tokens=0)), None, None, None,
                             ctypes.c_float(1e-6), None) == OK


def prologue(L, dims, **over):
    args = dict(xq=ctypes.c_void_p(0x100000), xk=ctypes.c_void_p(0x200000),
                xv=ctypes.c_void_p(0x300000), w=ctypes.c_void_p(0x400000), cin=None, cu=None,
                q=ctypes.c_void_p(0x500000), k=ctypes.c_void_p(0x600000),
                v=ctypes.c_void_p(0x700000), cout=None, eps=1e-6)
    args.update(over)
    d = None if dims is None else ctypes.byref(dims)
    return L.kda_qkv_prologue(d, args["xq"], args["xk"], args["xv"], args["w"], args["cin"],
                              args["cu"], args["q"], args["k"], args["v"], args["cout"],
                              ctypes.c_float(args["eps"]), None)


@pytest.mark.parametrize("dims,over,want", [
    (None, {}, INVALID), (D(num_heads=0), {}, INVALID),
    (D(d_k=96, d_v=96), {}, UNSUPPORTED),
    (D(num_seqs=3), {}, INVALID),                                   # 16 tokens, 3 sequences
    (D(), {"eps": 0.0}, INVALID), (D(), {"eps": float("nan")}, INVALID),
    (D(), {"eps": float("inf")}, INVALID),
    (D(), {"xk": None}, INVALID), (D(), {"v": None}, INVALID), (D(), {"w": None}, INVALID),
    (D(), {"xk": ctypes.c_void_p(0x200004)}, INVALID),             # bf16 x 4 needs 8 bytes
    (D(in_dtype=0), {"xk": ctypes.c_void_p(0x200008)}, INVALID),   # fp32 x 4 needs 16
    (D(), {"q": ctypes.c_void_p(0x500002)}, INVALID),
    (D(), {"w": ctypes.c_void_p(0x400008)}, INVALID),
    (D(), {"cin": ctypes.c_void_p(0x800008)}, INVALID),
    (D(), {"cout": ctypes.c_void_p(0x800002)}, INVALID),
    (D(), {"q": ctypes.c_void_p(0x100100)}, INVALID),              # q overlaps x_q
    (D(), {"k": ctypes.c_void_p(0x500000)}, INVALID),              # k is q
    (D(), {"v": ctypes.c_void_p(0x400010)}, INVALID),              # v overlaps the weights
    (D(), {"cin": ctypes.c_void_p(0x800000), "cout": ctypes.c_void_p(0x800100)}, INVALID),
    (D(), {"cout": ctypes.c_void_p(0x300000)}, INVALID),           # state out overlaps x_v
])
def test_qkv_prologue_rejects(L, dims, over, want):
    assert prologue(L, dims, **over) == want


def test_qkv_prologue_no_sequences_is_ok(L):
    # tokens but no sequence (cu_seqlens = [0]): nothing belongs to a sequence,
    # nothing is launched, cu_seqlens is not read past its one entry
    assert prologue(L, D(num_seqs=0, total_tokens=16), cu=ctypes.c_void_p(0x900000)) == OK


def test_qkv_prologue_empty_batch_is_ok(L):
    assert prologue(L, D(num_seqs=0, total_tokens=0), xq=None, xk=None, xv=None, w=None,
                    q=None, k=None, v=None) == OK


# Partial overlaps of an output with an input (or another output): each case
# moves one buffer so that it shares bytes with another; the rest of the call
# is valid, so the overlap is the only reason to reject it.
@pytest.mark.parametrize("over", [
    {"out": ctypes.c_void_p(0x10000 + 4096)},                   # out over the tail of q/k/v
    {"out": ctypes.c_void_p(0x10000 + 12288)},                  # out over the fp32 g only
    {"fin": ctypes.c_void_p(0x20000 + 256)},                    # final state over out
    {"init": ctypes.c_void_p(0x40000), "fin": ctypes.c_void_p(0x40000 - 64)},
    {"cu": ctypes.c_void_p(0x20000 + 64)},                      # out over cu_seqlens
])
def test_prefill_rejects_overlaps(L, over):
    base = dict(fin=None)
    base.update(over)
    assert prefill(L, D(), **base) == INVALID


def test_prefill_checkpoints_must_not_overlap_out(L):
    assert prefill_ckpt(L, D(), ckpt=ctypes.c_void_p(0x20000 - 1024)) == INVALID


@pytest.mark.parametrize("over", [
    {"dk": ctypes.c_void_p(0xa0000 + 4096)},                    # two gradients overlap
    {"dg": ctypes.c_void_p(0x1000000 + 8192)},                  # dg over the chunk states
    {"db": ctypes.c_void_p(0x98000 + 128)},                     # dbeta over d_out
    {"dinit": ctypes.c_void_p(0x10000)},                        # d_init over the inputs
])
def test_backward_rejects_overlaps(L, over):
    assert backward(L, D(), **over) == INVALID


@pytest.mark.parametrize("over", [
    {"out": ctypes.c_void_p(0x30000 + 1024)},                   # out inside the state
    {"state": ctypes.c_void_p(0x10000 - 256)},                  # state over q/k/v/g
])
def test_decode_rejects_overlaps(L, over):
    assert decode(L, D(num_seqs=4, total_tokens=4), **over) == INVALID


def test_output_gate_rejects_overlaps(L):
    # out (8 KB bf16 at 0x20000) over the norm weight
    assert L.kda_output_gate(ctypes.byref(D()), ctypes.c_void_p(0x20000),
                             ctypes.c_void_p(0x60000), ctypes.c_void_p(0x21000),
                             ctypes.c_float(1e-6), None) == INVALID


def test_checkpoint_count():
    cu = torch.tensor([0, 100, 164, 164, 364], dtype=torch.int32)
    assert kda.checkpoint_count(364, 32, cu) == 3 + 2 + 0 + 6
    assert kda.checkpoint_count(364, 64, cu) == 1 + 1 + 0 + 3
    assert kda.checkpoint_count(256, 64, None, num_seqs=2) == 4
    assert kda.checkpoint_count(0, 32, None, num_seqs=0) == 0


def test_prefill_empty_batch_is_ok(L):
    # nothing to do: no sequences, no tokens -> OK without touching the device
    assert prefill(L, D(num_seqs=0, total_tokens=0), q=None, k=None, v=None, g=None,
                   beta=None, out=None) == OK


@pytest.mark.parametrize("dims,over,want", [
    (D(num_seqs=4, total_tokens=5), {}, INVALID),           # one token per sequence
    (D(num_seqs=4, total_tokens=4, d_k=64, d_v=128), {}, UNSUPPORTED),
    (D(num_seqs=4, total_tokens=4), {"state": None}, INVALID),
    (D(num_seqs=4, total_tokens=4), {"state": FAKE_MISALIGNED}, INVALID),
    (D(num_seqs=4, total_tokens=4), {"out": ctypes.c_void_p(0x30000)}, INVALID),
    (D(num_seqs=4, total_tokens=4), {"k": None}, INVALID),
])
def test_decode_rejects(L, dims, over, want):
    assert decode(L, dims, **over) == want


def test_decode_empty_is_ok(L):
    assert decode(L, D(num_seqs=0, total_tokens=0)) == OK


def test_python_binding_rejects_cpu_tensors():
    x = torch.zeros(4, 1, 64)
    with pytest.raises(ValueError):
        kda.kda_prefill(x, x, x, x, torch.zeros(4, 1))
