"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (default variant, whole batch in one call).  Every (sequence,
head) pair is independent, so the oracle checks all of them where it finishes
in seconds (the 8K prefill, the decode workload), every sequence with a
quarter of the heads for the packed varlen batch, and 16 heads over the whole
length of the 262,144-token context (host memory and the oracle's minutes
bound the rest)."""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth
import oracle
from kda_testutil import TOL, rel_err, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu(inp, out_dtype):
    return kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           init_state=inp["init_state"], cu_seqlens=inp["cu_seqlens"],
                           out_dtype=out_dtype)


def test_prefill_8k_all_heads():
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, DEV)
    out32, fin32 = _gpu(inp, torch.float32)
    out16, fin16 = _gpu(inp, torch.bfloat16)
    assert torch.equal(out16, out32.to(torch.bfloat16))
    assert torch.equal(fin16, fin32)
    o_ref, s_ref = oracle.prefill(*(host64(inp[x]) for x in ("q", "k", "v", "g", "beta")))
    eo, es = rel_err(host64(out32), o_ref), rel_err(host64(fin32), s_ref)
    print(f"prefill_8k: err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]


def _oracle_heads(inp, n, heads):
    """The oracle on sequence n for the given heads, in one threaded call."""
    cu = inp["cu_seqlens"].cpu().numpy()
    sl = slice(int(cu[n]), int(cu[n + 1]))
    args = [host64(inp[x][sl][:, heads]) for x in ("q", "k", "v", "g", "beta")]
    init = None if inp["init_state"] is None else host64(inp["init_state"][n:n + 1][:, heads])
    o, s = oracle.prefill(*args, init_state=init, num_threads=oracle.num_cpus())
    return sl, o, s[0]


def test_varlen_packed_every_sequence():
    """All eight sequences of the packed batch (nonzero initial states), 24 of
    the 96 heads each (every fourth head), against the oracle."""
    w = synth.WORKLOADS["varlen_8seq"]
    inp = synth.prefill_inputs(w, DEV)
    out32, fin32 = _gpu(inp, torch.float32)
    heads = list(range(0, w.heads, 4))
    g_o, g_s, o_all, s_all = [], [], [], []
    for n in range(w.num_seqs):
        sl, o, s = _oracle_heads(inp, n, heads)
        o_all.append(o.reshape(-1)); s_all.append(s.reshape(-1))
        g_o.append(host64(out32[sl][:, heads]).reshape(-1))
        g_s.append(host64(fin32[n][heads]).reshape(-1))
    eo = rel_err(np.concatenate(g_o), np.concatenate(o_all))
    es = rel_err(np.concatenate(g_s), np.concatenate(s_all))
    print(f"varlen_8seq (8 sequences x 24 heads): err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]


def test_prefill_256k_sixteen_heads():
    """The 262,144-token context (long retention, x ~ N(4, 1)): 16 heads spread
    over the 96, each over its whole length."""
    w = synth.WORKLOADS["prefill_256k"]
    inp = synth.prefill_inputs(w, DEV)
    out32, fin32 = _gpu(inp, torch.float32)
    heads = list(range(0, w.heads, 6))
    sl, o, s = _oracle_heads(inp, 0, heads)
    eo = rel_err(host64(out32[sl][:, heads]), o)
    es = rel_err(host64(fin32[0][heads]), s)
    print(f"prefill_256k (16 heads): err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]
    assert torch.isfinite(out32).all() and torch.isfinite(fin32).all()


def test_decode_256x64_all_pairs():
    w = synth.WORKLOADS["decode_256x64"]
    x = synth.decode_inputs(w, DEV)
    st = x["state"].clone()
    ref = host64(x["state"])
    outs, refs = [], []
    for s in range(w.steps):
        out = kda.kda_decode(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], st,
                             out_dtype=torch.float32)
        o_ref, ref = oracle.decode(*(host64(x[n][s]) for n in ("q", "k", "v", "g", "beta")), ref,
                                   inplace=True)
        outs.append(host64(out)); refs.append(o_ref)
    eo = rel_err(np.stack(outs), np.stack(refs))
    es = rel_err(host64(st), ref)
    print(f"decode_256x64: err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]


def test_prefill_8k_checkpoints_match_prefix_runs():
    """Full-size layer with a checkpoint every 1024 tokens: the outputs equal
    the plain prefill's, and checkpoints 1, 4 and 8 equal (bitwise) the final
    states of prefills over the first 1024, 4096 and 8192 tokens."""
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, "cuda")
    out, fin, ck = kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"],
                                                inp["beta"], cu_seqlens=inp["cu_seqlens"],
                                                interval=1024)
    assert ck.shape == (8, w.heads, w.d, w.d)
    out0, fin0 = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 cu_seqlens=inp["cu_seqlens"])
    assert torch.equal(out, out0) and torch.equal(fin, fin0)
    assert torch.equal(ck[7], fin0[0])
    for j in (1, 4):
        n = 1024 * j
        _, fin_p = kda.kda_prefill(*(inp[x][:n].contiguous() for x in ("q", "k", "v", "g", "beta")))
        assert torch.equal(ck[j - 1], fin_p[0]), f"checkpoint {j}"


def test_gated_prefill_8k_sampled_heads():
    """The 8K layer through the fused gate prologue (bf16 decay logits):
    three heads against the oracle fed with the oracle's gate."""
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, "cuda")
    gl = synth.gate_logits(w.total_tokens, w.heads, w.d, dtype=w.dtype, seed=81, device="cuda")
    out, fin = kda.kda_prefill_gated(inp["q"], inp["k"], inp["v"], gl["z"], gl["a_log"],
                                     gl["beta_logit"], cu_seqlens=inp["cu_seqlens"],
                                     out_dtype=torch.float32)
    heads = [0, 47, 95]
    g, beta = oracle.gate(host64(gl["z"][:, heads]), host64(gl["a_log"][heads]),
                          host64(gl["beta_logit"][:, heads]))
    o_ref, s_ref = oracle.prefill(host64(inp["q"][:, heads]), host64(inp["k"][:, heads]),
                                  host64(inp["v"][:, heads]), g, beta)
    eo = rel_err(host64(out[:, heads]), o_ref)
    es = rel_err(host64(fin[:, heads]), s_ref)
    print(f"gated prefill_8k (3 heads): err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]


def test_output_gated_8k_sampled_heads():
    """The 8K layer through kda_prefill_output_gated (bf16 out, the launch the
    benchmark times: the prefill, then the gate in place): three heads against
    the oracle's prefill followed by the oracle's output gate."""
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, "cuda")
    og = synth.output_gate_inputs(w.total_tokens, w.heads, w.d, dtype=w.dtype, seed=83,
                                  device="cuda")
    eps = 1e-6
    out, fin = kda.kda_prefill_output_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                            og["gate"], og["norm_weight"], eps,
                                            cu_seqlens=inp["cu_seqlens"])
    assert out.dtype == torch.bfloat16
    heads = [0, 47, 95]
    o_ref, s_ref = oracle.prefill(*(host64(inp[x][:, heads]) for x in ("q", "k", "v", "g", "beta")))
    y_ref = oracle.output_gate(o_ref, host64(og["gate"][:, heads]), host64(og["norm_weight"]), eps)
    eo = rel_err(host64(out[:, heads]), y_ref)
    es = rel_err(host64(fin[:, heads]), s_ref)
    bound = TOL[torch.bfloat16] + 2.0 ** -8 * np.abs(y_ref).max() / np.sqrt(np.mean(y_ref ** 2))
    print(f"output-gated prefill_8k (3 heads, bf16 out): err_y {eo:.3e} (bound {bound:.3e}) "
          f"err_S {es:.3e}")
    assert eo <= bound and es <= TOL[torch.bfloat16]


def test_scalar_decay_8k_sampled_heads():
    """The 8K layer as Gated DeltaNet (one decay per head and step), in the
    launch the benchmark times: three heads against the oracle."""
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, "cuda")
    gh = synth.scalar_decay(w.total_tokens, w.heads, seed=85, device="cuda")
    out, fin = kda.kda_prefill_scalar_decay(inp["q"], inp["k"], inp["v"], gh, inp["beta"],
                                            cu_seqlens=inp["cu_seqlens"], out_dtype=torch.float32)
    heads = [0, 47, 95]
    o_ref, s_ref = oracle.prefill_scalar_decay(
        *(host64(inp[x][:, heads]) for x in ("q", "k", "v")), host64(gh[:, heads]),
        host64(inp["beta"][:, heads]))
    eo = rel_err(host64(out[:, heads]), o_ref)
    es = rel_err(host64(fin[:, heads]), s_ref)
    print(f"scalar-decay prefill_8k (3 heads): err_o {eo:.3e} err_S {es:.3e}")
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]
