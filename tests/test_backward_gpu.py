"""GPU parity of kda_backward (the gradients of the chunked prefill) with the
oracle's reverse mode through the token recurrence."""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth
import oracle
from kda_testutil import TOL, rel_err, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "d_init_state")


def _upstream(T, H, N, d, dtype, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    d_out = torch.randn((T, H, d), generator=gen, device=DEV).to(dtype)
    d_fin = 0.5 * torch.randn((N, H, d, d), generator=gen, device=DEV)
    return d_out, d_fin


def _oracle_grads(inp, d_out, d_fin, cu, heads=None):
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads])
    return oracle.backward(*(host64(sel(inp[x])) for x in ("q", "k", "v", "g", "beta")),
                           host64(sel(d_out)),
                           None if d_fin is None else host64(d_fin if heads is None else d_fin[:, heads]),
                           init_state=None if inp.get("init_state") is None else
                           host64(inp["init_state"] if heads is None else inp["init_state"][:, heads]),
                           cu_seqlens=None if cu is None else cu.cpu().numpy())


def _check(res, ref, tol, heads=None):
    errs = {}
    for name in GRADS:
        x = host64(res[name])
        if heads is not None:
            x = x[:, heads]
        errs[name] = rel_err(x, ref[name])
    bad = {k: v for k, v in errs.items() if v > tol}
    assert not bad, f"gradient errors above {tol}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_matches_oracle(d, dtype):
    """A ragged packed batch (one token, chunk-1, chunk, chunk+1, empty, multi-
    chunk) with initial states and final-state gradients; the chunk states come
    from kda_prefill_checkpointed with interval CHUNK (tensor cores for bf16,
    d = 128)."""
    H = 2
    lens = [1, 31, 32, 33, 0, 65, 100]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=111, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    d_out, d_fin = _upstream(T, H, len(lens), d, dtype, 112)
    res = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                           init_state=inp["init_state"], cu_seqlens=cu, grad_dtype=torch.float32)
    ref = _oracle_grads(inp, d_out, d_fin, cu)
    errs = _check(res, ref, TOL[dtype])
    print(f"backward d={d} {dtype}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))


def test_backward_bf16_grads_are_rne_of_fp32():
    T, H, d = 100, 2, 128
    inp = synth.random_inputs(T, H, d, dtype=torch.bfloat16, seed=113, device=DEV)
    d_out, d_fin = _upstream(T, H, 1, d, torch.bfloat16, 114)
    a = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                         grad_dtype=torch.float32)
    b = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                         grad_dtype=torch.bfloat16)
    for name in ("dq", "dk", "dv"):
        assert torch.equal(b[name], a[name].to(torch.bfloat16)), name
    for name in ("dg", "dbeta", "d_init_state"):
        assert torch.equal(b[name], a[name]), name


def test_backward_single_chunks_need_no_states():
    """Sequences of at most one chunk: no chunk states, no d_final; the
    gradients still match the oracle."""
    H, d = 3, 64
    lens = [5, 20, 7]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=torch.float32, seed=115, device=DEV)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    d_out, _ = _upstream(T, H, len(lens), d, torch.float32, 116)
    res = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                           cu_seqlens=cu, chunk_states=torch.empty((0, H, d, d), device=DEV))
    ref = _oracle_grads(inp, d_out, None, cu)
    _check(res, ref, TOL[torch.float32])


def test_backward_layer_1k_sampled_heads():
    """The 96-head layer over 1024 tokens (bf16, tensor-core forward states),
    in one launch; three heads against the oracle."""
    T, H, d = 1024, 96, 128
    inp = synth.random_inputs(T, H, d, dtype=torch.bfloat16, seed=117, device=DEV)
    d_out, d_fin = _upstream(T, H, 1, d, torch.bfloat16, 118)
    res = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                           grad_dtype=torch.float32)
    heads = [0, 47, 95]
    ref = _oracle_grads(inp, d_out, d_fin, None, heads=heads)
    errs = _check(res, ref, TOL[torch.bfloat16], heads=heads)
    print("backward 1k layer (3 heads): " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))


def test_backward_8k_layer_sampled_heads():
    """The 8K layer's gradients in the launch the benchmark times (all 96 heads,
    chunk states from the tensor-core forward): two heads against the oracle's
    reverse mode over all 8192 tokens (which keeps every state: about 1 GB of
    host memory per head)."""
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, DEV)
    T, H, d = inp["q"].shape
    d_out, d_fin = _upstream(T, H, 1, d, w.dtype, 119)
    res = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                           cu_seqlens=inp["cu_seqlens"], grad_dtype=torch.float32)
    heads = [0, 95]
    ref = _oracle_grads(inp, d_out, d_fin, None, heads=heads)
    errs = _check(res, ref, TOL[torch.bfloat16], heads=heads)
    print("backward 8k layer (2 heads): " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))


def test_missing_chunk_states_are_reported():
    """Chunk-state rows past chunk_capacity: rejected on the host when the lengths
    are known there (no cu_seqlens), reported by the device status otherwise."""
    dev = "cuda"
    inp = synth.random_inputs(96, 2, 128, dtype=torch.bfloat16, seed=31, device=dev)
    gen = torch.Generator(device=dev).manual_seed(32)
    d_out = torch.randn(inp["q"].shape, generator=gen, device=dev).to(torch.bfloat16)
    _, _, cs = kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                            interval=kda.CHUNK)
    short = cs[:1].contiguous()   # 96 tokens need 2 rows (the starts of chunks 1 and 2)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                         chunk_states=short)
    assert e.value.status == 1
    cu = torch.tensor([0, 96], dtype=torch.int32, device=dev)
    kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                     cu_seqlens=cu, chunk_states=short)
    assert kda.kda_get_last_device_error() == 1      # KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_get_last_device_error() == 0      # cleared by the read
    kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                     cu_seqlens=cu, chunk_states=cs)
    assert kda.kda_get_last_device_error() == 0


def test_backward_bf16_unaligned_gradients_match_aligned():
    """The tensor-core backward writes bf16 gradient rows through shared memory as
    16-byte stores when the gradient arrays are 16-byte aligned, and element by
    element otherwise: both give the same bits (a ragged packed batch, so that the
    last chunk of a sequence is partial)."""
    import ctypes
    H, d = 2, 128
    lens = [70, 33, 96]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=torch.bfloat16, seed=121, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    d_out, d_fin = _upstream(T, H, len(lens), d, torch.bfloat16, 122)
    ref = kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out, d_fin,
                           init_state=inp["init_state"], cu_seqlens=cu)
    _, _, cst = kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                             inp["init_state"], cu, interval=kda.CHUNK)
    n = T * H * d
    # each gradient 2 elements (4 or 8 bytes) past a 16-byte boundary
    bufs = {name: torch.zeros(n + 8, dtype=dt, device=DEV)
            for name, dt in (("dq", torch.bfloat16), ("dk", torch.bfloat16), ("dv", torch.bfloat16),
                             ("dg", torch.float32))}
    views = {name: b[2:2 + n].view(T, H, d) for name, b in bufs.items()}
    dbeta = torch.empty((T, H), dtype=torch.float32, device=DEV)
    dinit = torch.empty((len(lens), H, d, d), dtype=torch.float32, device=DEV)
    dims = kda.Dims(len(lens), T, H, d, d, kda._DTYPES[torch.bfloat16], kda._DTYPES[torch.bfloat16], 0)
    p = lambda x: ctypes.c_void_p(x.data_ptr()) if x is not None else None
    st = kda.lib().kda_backward(ctypes.byref(dims), p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["g"]),
                                p(inp["beta"]), p(inp["init_state"]), p(cu), p(cst), int(cst.shape[0]),
                                p(d_out), p(d_fin), p(views["dq"]), p(views["dk"]), p(views["dv"]),
                                p(views["dg"]), p(dbeta), p(dinit), None)
    assert st == 0
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_error() == 0
    for name in ("dq", "dk", "dv", "dg"):
        assert torch.equal(views[name], ref[name]), name
    assert torch.equal(dbeta, ref["dbeta"]) and torch.equal(dinit, ref["d_init_state"])
