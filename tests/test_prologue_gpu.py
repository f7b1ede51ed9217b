"""GPU parity of the q, k, v prologue (ShortConv width 4, Swish, L2Norm of q
and k) through the C ABI against the fp64 oracle: a ragged packed batch with
empty and short sequences, both head sizes, every dtype pair, with and without
a carried conv state; the conv state carried across calls (a decode step is a
one-token call) bit-for-bit; the 8K-token, 96-head layer on sampled heads;
windows of the 262,144-token layer on all heads.

Bounds, elementwise: the kernel computes in fp32 (four fused multiply-adds,
one fast exponential, one division, a 128-term sum of squares and a
reciprocal square root), so an fp32 output is within 1e-5 |ref| + 2e-6 rms of
the exact result; a bf16 output is that value rounded to nearest, within
2^-8 |ref| more.  The conv state out holds copies of inputs: exact."""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth
import oracle
from kda_testutil import host64

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16


def bound(ref, out_dtype):
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    rel = 1e-5 + (2.0 ** -8 if out_dtype == BF16 else 0.0)
    return rel * np.abs(ref) + 2e-6 * rms


def check_against_oracle(p, cu, state, outs, eps=1e-6):
    ref = oracle.qkv_prologue(host64(p["x_q"]), host64(p["x_k"]), host64(p["x_v"]),
                              host64(p["conv_weight"]),
                              cu_seqlens=None if cu is None else cu.cpu().numpy(),
                              conv_state=host64(state), eps=eps)
    worst = 0.0
    for name, got, want in zip("qkv", outs[:3], ref[:3]):
        g = host64(got)
        err = np.abs(g - want)
        lim = bound(want, got.dtype)
        assert np.all(err <= lim), (
            f"{name}: max excess {np.max(err - lim):.3e}, max |err| {err.max():.3e}")
        worst = max(worst, float(err.max()))
    if outs[3] is not None:
        assert np.array_equal(host64(outs[3]), ref[3]), "conv state out differs"
    return worst


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("in_dtype,out_dtype", [(F32, F32), (BF16, BF16), (BF16, F32),
                                                (F32, BF16)])
@pytest.mark.parametrize("with_state", [False, True])
def test_ragged_batch_matches_oracle(d, in_dtype, out_dtype, with_state):
    lens = [37, 0, 5, 130, 1, 2, 64]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    T, H, N = int(sum(lens)), 3, len(lens)
    p = synth.qkv_projections(T, H, d, N=N, dtype=in_dtype, seed=40 + d, device=DEV)
    state = p["conv_state"] if with_state else None
    outs = kda.kda_qkv_prologue(p["x_q"], p["x_k"], p["x_v"], p["conv_weight"], cu_seqlens=cu,
                                conv_state=state, out_dtype=out_dtype)
    torch.cuda.synchronize()
    check_against_oracle(p, cu, state, outs)


def test_equal_length_layout_and_tail():
    """cu_seqlens = NULL (equal sequences), a length that is not a multiple
    of the 16-token tile."""
    N, L, H, d = 3, 21, 2, 128
    p = synth.qkv_projections(N * L, H, d, N=N, dtype=BF16, seed=47, device=DEV)
    outs = kda.kda_qkv_prologue(p["x_q"], p["x_k"], p["x_v"], p["conv_weight"], num_seqs=N,
                                conv_state=p["conv_state"])
    cu = torch.arange(0, N * L + 1, L, dtype=torch.int32, device=DEV)
    check_against_oracle(p, cu, p["conv_state"], outs)


def test_decode_steps_equal_one_call():
    """One call over whole sequences equals one-token calls (num_seqs tokens
    each) that carry the conv state, bit for bit: the taps see the same
    values in the same order."""
    N, L, H, d = 4, 9, 2, 128
    p = synth.qkv_projections(N * L, H, d, N=N, dtype=BF16, seed=48, device=DEV)
    xs = [p[n].view(N, L, H, d) for n in ("x_q", "x_k", "x_v")]
    whole = kda.kda_qkv_prologue(*(x.reshape(N * L, H, d) for x in xs), p["conv_weight"],
                                 num_seqs=N, conv_state=p["conv_state"])
    st = [p["conv_state"].clone(), torch.empty_like(p["conv_state"])]
    for i in range(L):
        step = kda.kda_qkv_prologue(*(x[:, i].contiguous() for x in xs), p["conv_weight"],
                                    num_seqs=N, conv_state=st[i % 2],
                                    conv_state_out=st[(i + 1) % 2])
        for a, b in zip(step[:3], whole[:3]):
            assert torch.equal(a, b.view(N, L, H, d)[:, i])
    assert torch.equal(st[L % 2], whole[3])


def test_split_call_carries_the_state():
    """A sequence cut in two: the second call takes the first call's conv
    state out and gives what one call gives, bit for bit."""
    T, T1, H, d = 100, 37, 2, 64
    p = synth.qkv_projections(T, H, d, dtype=F32, seed=49, device=DEV)
    whole = kda.kda_qkv_prologue(p["x_q"], p["x_k"], p["x_v"], p["conv_weight"],
                                 conv_state=p["conv_state"])
    a = kda.kda_qkv_prologue(p["x_q"][:T1], p["x_k"][:T1], p["x_v"][:T1], p["conv_weight"],
                             conv_state=p["conv_state"])
    b = kda.kda_qkv_prologue(p["x_q"][T1:], p["x_k"][T1:], p["x_v"][T1:], p["conv_weight"],
                             conv_state=a[3])
    for i in range(3):
        assert torch.equal(torch.cat([a[i], b[i]]), whole[i])
    assert torch.equal(b[3], whole[3])


def test_state_only_call():
    """No tokens: the call only moves the conv state (each sequence's last
    three inputs are the state in)."""
    N, H, d = 3, 2, 64
    p = synth.qkv_projections(1, H, d, N=N, dtype=F32, seed=50, device=DEV)
    cu = torch.zeros(N + 1, dtype=torch.int32, device=DEV)
    e = torch.empty((0, H, d), device=DEV)
    out = kda.kda_qkv_prologue(e, e, e, p["conv_weight"], cu_seqlens=cu,
                               conv_state=p["conv_state"])
    assert torch.equal(out[3], p["conv_state"])
    out = kda.kda_qkv_prologue(e, e, e, p["conv_weight"], cu_seqlens=cu)
    assert torch.all(out[3] == 0)


def test_zero_rows_stay_finite():
    """An all-zero projection gives zero q, k, v (eps keeps the norm finite)."""
    T, H, d = 20, 2, 128
    p = synth.qkv_projections(T, H, d, dtype=BF16, seed=51, device=DEV)
    z = torch.zeros_like(p["x_q"])
    q, k, v, _ = kda.kda_qkv_prologue(z, z, z, p["conv_weight"])
    for t in (q, k, v):
        assert torch.all(t == 0)


def test_layer_8k_sampled_heads():
    """The 8K-token, 96-head layer (bf16 in and out, the benchmark's launch),
    compared on eight heads (heads are independent, so slicing them out of
    the inputs gives the oracle the exact same problem)."""
    T, H, d = 8192, 96, 128
    p = synth.qkv_projections(T, H, d, dtype=BF16, seed=52, device=DEV)
    q, k, v, cs = kda.kda_qkv_prologue(p["x_q"], p["x_k"], p["x_v"], p["conv_weight"])
    torch.cuda.synchronize()
    heads = [0, 13, 27, 40, 55, 68, 81, 95]
    sub = {n: p[n][:, heads].contiguous() for n in ("x_q", "x_k", "x_v")}
    sub["conv_weight"] = p["conv_weight"][:, heads].contiguous()
    outs = (q[:, heads], k[:, heads], v[:, heads], cs[:, :, :, heads])
    check_against_oracle(sub, None, None, outs)


def test_layer_256k_sampled_windows():
    """The longest workload's shapes (262,144 tokens, 96 heads, bf16; 38.7 GB
    in and out).  The convolution looks back three tokens only, so a window
    [t0, t0 + 48) is exactly the oracle's run over that window with the three
    inputs before it as the carried state.  Windows at the start, at a tile
    edge, in the middle and at the end, on all heads."""
    T, H, d = 262144, 96, 128
    p = synth.qkv_projections(T, H, d, dtype=BF16, seed=53, device=DEV)
    q, k, v, cs = kda.kda_qkv_prologue(p["x_q"], p["x_k"], p["x_v"], p["conv_weight"])
    torch.cuda.synchronize()
    for t0 in (0, 4096 * 16 + 13, 131072, T - 48):
        t1 = t0 + 48
        sub = {n: p[n][t0:t1] for n in ("x_q", "x_k", "x_v")}
        sub["conv_weight"] = p["conv_weight"]
        state = torch.zeros((1, 3, 3, H, d), device=DEV)
        for si, n in enumerate(("x_q", "x_k", "x_v")):
            for j in range(3):
                u = t0 - 3 + j
                if u >= 0:
                    state[0, si, j] = p[n][u].float()
        outs = (q[t0:t1], k[t0:t1], v[t0:t1], cs if t1 == T else None)
        check_against_oracle(sub, None, state, outs)
    del p, q, k, v, cs
    torch.cuda.empty_cache()
