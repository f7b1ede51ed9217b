"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle, on
sizes the oracle finishes in seconds: several chunks, ragged tails, empty
sequences, both head sizes, both input dtypes, every prefill variant."""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth
import oracle
from kda_testutil import TOL, rel_err, host64

pytestmark = pytest.mark.gpu

DEV = "cuda"
VARIANTS = [kda.PREFILL_DEFAULT, kda.PREFILL_FP32, kda.PREFILL_TC, kda.PREFILL_TC_SPLIT,
            kda.PREFILL_TC_2PASS]


def supported(variant, d, dtype):
    """The tensor-core kernel takes d = 128 with bf16 inputs only (its tf32
    operands cannot meet the 1e-4 bound of fp32 inputs)."""
    if variant in (kda.PREFILL_TC, kda.PREFILL_TC_SPLIT, kda.PREFILL_TC_2PASS):
        return d == 128 and dtype == torch.bfloat16
    return True


def run_gpu(inp, variant, out_dtype=torch.float32, cu=None, num_seqs=None):
    try:
        return kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               init_state=inp.get("init_state"), cu_seqlens=cu,
                               num_seqs=num_seqs, out_dtype=out_dtype, variant=variant)
    except kda.KdaError as e:
        if e.status == 2:
            pytest.skip("variant does not take this shape/dtype (KDA_ERR_UNSUPPORTED)")
        raise


def run_oracle(inp, cu=None, num_seqs=None):
    return oracle.prefill(host64(inp["q"]), host64(inp["k"]), host64(inp["v"]), host64(inp["g"]),
                          host64(inp["beta"]), init_state=host64(inp.get("init_state")),
                          cu_seqlens=None if cu is None else cu.cpu().numpy(),
                          num_seqs=num_seqs)


def check(out, fin, o_ref, s_ref, dtype):
    eo = rel_err(host64(out), o_ref)
    es = rel_err(host64(fin), s_ref)
    assert eo <= TOL[dtype], f"output error {eo:.3e} > {TOL[dtype]}"
    assert es <= TOL[dtype], f"final-state error {es:.3e} > {TOL[dtype]}"
    return eo, es


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_fp32_workload(variant):
    """The small fp32 workload (T=256, H=2, d=64) in full, at 1e-4."""
    w = synth.WORKLOADS["tiny_fp32"]
    if not supported(variant, w.d, w.dtype):
        pytest.skip("variant does not take d=64")
    inp = synth.prefill_inputs(w, DEV)
    out, fin = run_gpu(inp, variant)
    o_ref, s_ref = run_oracle(inp)
    check(out, fin, o_ref, s_ref, torch.float32)


LENS = [1, 31, 32, 33, 0, 64, 65, 100, 257, 16, 15]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_packed_batch(variant, d, dtype):
    """Packed sequences whose lengths straddle every chunk boundary, with a
    nonzero initial state and empty sequences in the middle."""
    if not supported(variant, d, dtype):
        pytest.skip("variant does not take this head size")
    T = sum(LENS)
    inp = synth.random_inputs(T, 3, d, dtype=dtype, seed=d + (dtype == torch.bfloat16),
                              device=DEV, num_seqs=len(LENS), init_std=0.05)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(LENS)]), dtype=torch.int32, device=DEV)
    out, fin = run_gpu(inp, variant, cu=cu)
    o_ref, s_ref = run_oracle(inp, cu=cu)
    check(out, fin, o_ref, s_ref, dtype)
    init = inp["init_state"].cpu()
    for n, L in enumerate(LENS):
        if L == 0:
            assert torch.equal(fin[n].cpu(), init[n]), "empty sequence must carry its state"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_bf16_out_is_rne_of_fp32_out(variant, dtype):
    if not supported(variant, 128, dtype):
        pytest.skip("variant does not take this case")
    inp = synth.random_inputs(300, 4, 128, dtype=dtype, seed=7, device=DEV)
    o32, f32 = run_gpu(inp, variant, torch.float32)
    o16, f16 = run_gpu(inp, variant, torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(f16, f32)


@pytest.mark.parametrize("variant", VARIANTS)
def test_equal_length_layout_without_cu(variant):
    inp = synth.random_inputs(4 * 70, 2, 128, dtype=torch.bfloat16, seed=3, device=DEV,
                              num_seqs=4, init_std=0.02)
    out, fin = run_gpu(inp, variant, num_seqs=4)
    o_ref, s_ref = run_oracle(inp, num_seqs=4)
    check(out, fin, o_ref, s_ref, torch.bfloat16)


@pytest.mark.parametrize("variant", VARIANTS)
def test_final_state_may_alias_init(variant):
    inp = synth.random_inputs(90, 2, 128, dtype=torch.bfloat16, seed=5, device=DEV,
                              init_std=0.05)
    out_a, fin_a = run_gpu(inp, variant)
    st = inp["init_state"].clone()
    out_b, _ = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               init_state=st, final_state=st, out_dtype=torch.float32,
                               variant=variant)
    assert torch.equal(out_a, out_b)
    assert torch.equal(fin_a, st)


@pytest.mark.parametrize("variant", VARIANTS)
def test_final_state_may_alias_init_packed(variant):
    """In place over a packed batch of several multi-chunk sequences: every
    (sequence, head) slice is read before it is overwritten."""
    lens = [70, 33, 130, 0, 64]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    inp = synth.random_inputs(sum(lens), 3, 128, dtype=torch.bfloat16, seed=9, device=DEV,
                              num_seqs=len(lens), init_std=0.05)
    out_a, fin_a = run_gpu(inp, variant, cu=cu)
    st = inp["init_state"].clone()
    out_b, _ = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               init_state=st, final_state=st, cu_seqlens=cu,
                               out_dtype=torch.float32, variant=variant)
    assert torch.equal(out_a, out_b)
    assert torch.equal(fin_a, st)


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_tokens_copies_state(variant):
    N, H, d = 3, 2, 128
    init = torch.randn(N, H, d, d, device=DEV)
    e = torch.empty(0, H, d, device=DEV, dtype=torch.bfloat16)
    cu = torch.zeros(N + 1, dtype=torch.int32, device=DEV)
    inp = dict(q=e, k=e, v=e, g=e.float(), beta=torch.empty(0, H, device=DEV), init_state=init)
    _, fin = run_gpu(inp, variant, cu=cu)
    assert torch.equal(fin, init)
    inp["init_state"] = None
    _, fin0 = run_gpu(inp, variant, cu=cu)
    assert torch.count_nonzero(fin0) == 0


@pytest.mark.parametrize("variant", VARIANTS)
def test_out_of_range_cu_seqlens_is_clamped(variant):
    """cu entries beyond T_tot are clamped and a decreasing pair is empty."""
    T, H, d = 50, 2, 128
    inp = synth.random_inputs(T, H, d, dtype=torch.bfloat16, seed=11, device=DEV, num_seqs=3,
                              init_std=0.05)
    cu = torch.tensor([0, 50, 30, 999], dtype=torch.int32, device=DEV)
    out, fin = run_gpu(inp, variant, cu=cu)
    # sequence 0 covers [0, 50); sequence 1 (50 -> 30) is empty; sequence 2 is [30, 50)
    o0, s0 = oracle.prefill(*(host64(inp[x]) for x in ("q", "k", "v", "g", "beta")),
                            init_state=host64(inp["init_state"][:1]))
    assert rel_err(host64(fin[0]), s0[0]) <= TOL[torch.bfloat16]
    assert torch.equal(fin[1], inp["init_state"][1])
    sl = slice(30, 50)
    _, s2 = oracle.prefill(*(host64(inp[x][sl]) for x in ("q", "k", "v", "g", "beta")),
                           init_state=host64(inp["init_state"][2:3]))
    assert rel_err(host64(fin[2]), s2[0]) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_q_equals_k_beta_one_reads_v(variant, dtype):
    """Closed form: with beta = 1, q = k and unit keys, each token reads back
    exactly the value it wrote (the delta rule's beta = 1 property).  bf16
    keys are unit-norm only to about 2^-8, which the bf16 bound covers."""
    if not supported(variant, 128, dtype):
        pytest.skip("variant does not take this dtype")
    inp = synth.random_inputs(777, 4, 128, dtype=dtype, seed=13, device=DEV,
                              init_std=0.1)
    inp["q"] = inp["k"]
    inp["beta"] = torch.ones_like(inp["beta"])
    out, _ = run_gpu(inp, variant)
    assert rel_err(host64(out), host64(inp["v"])) <= TOL[dtype]


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_steps_match_oracle(d, dtype):
    N, H, S = 5, 3, 9
    st0 = torch.randn(N, H, d, d, device=DEV) * 0.05
    steps = [synth.random_inputs(N, H, d, dtype=dtype, seed=100 + s, device=DEV) for s in range(S)]
    st = st0.clone()
    ref = host64(st0)
    for s in range(S):
        x = steps[s]
        out = kda.kda_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], st,
                             out_dtype=torch.float32)
        o_ref, ref = oracle.decode(*(host64(x[n]) for n in ("q", "k", "v", "g", "beta")), ref)
        assert rel_err(host64(out), o_ref) <= TOL[dtype]
    assert rel_err(host64(st), ref) <= TOL[dtype]


def test_decode_bf16_out_is_rne_of_fp32_out():
    N, H, d = 7, 4, 128
    x = synth.random_inputs(N, H, d, dtype=torch.bfloat16, seed=3, device=DEV)
    st = torch.randn(N, H, d, d, device=DEV) * 0.05
    s1, s2 = st.clone(), st.clone()
    o32 = kda.kda_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], s1, out_dtype=torch.float32)
    o16 = kda.kda_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], s2, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(s1, s2)


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_equals_decode_steps(variant):
    """Prefill over T tokens equals T single-token decode updates."""
    T, H, d = 70, 2, 128
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=21, device=DEV, init_std=0.05)
    out, fin = run_gpu(inp, variant)
    st = inp["init_state"].clone()
    outs = []
    for t in range(T):
        sl = slice(t, t + 1)
        outs.append(kda.kda_decode(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["g"][sl],
                                   inp["beta"][sl], st, out_dtype=torch.float32))
    dec = torch.cat(outs)
    tol = TOL[dtype]
    assert rel_err(host64(out), host64(dec)) <= tol
    assert rel_err(host64(fin), host64(st)) <= tol


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("split", [97, 128])
def test_split_sequence_carries_state(variant, split):
    """Prefill over [0, T) equals prefill over [0, T1) followed by prefill over
    [T1, T) started from the first call's final state (chunk-aligned and
    ragged split points)."""
    T, H, d = 300, 2, 128
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=31, device=DEV, init_std=0.05)
    out, fin = run_gpu(inp, variant)
    a = {x: inp[x][:split].contiguous() for x in ("q", "k", "v", "g", "beta")}
    b = {x: inp[x][split:].contiguous() for x in ("q", "k", "v", "g", "beta")}
    a["init_state"] = inp["init_state"]
    out_a, fin_a = run_gpu(a, variant)
    b["init_state"] = fin_a
    out_b, fin_b = run_gpu(b, variant)
    tol = TOL[dtype]
    assert rel_err(host64(torch.cat([out_a, out_b])), host64(out)) <= tol
    assert rel_err(host64(fin_b), host64(fin)) <= tol


@pytest.mark.parametrize("variant", VARIANTS)
def test_packed_batch_equals_sequences_run_alone(variant):
    """A packed batch gives, for every sequence, exactly what that sequence
    gives alone: each (sequence, head) is computed independently and the same
    way whatever its position in the packed batch."""
    H, d = 2, 128
    lens = [45, 96, 1, 130]
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=41, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    out, fin = run_gpu(inp, variant, cu=cu)
    for n, (t0, t1) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        one = {x: inp[x][t0:t1].contiguous() for x in ("q", "k", "v", "g", "beta")}
        one["init_state"] = inp["init_state"][n:n + 1].contiguous()
        o1, f1 = run_gpu(one, variant)
        assert torch.equal(o1, out[t0:t1]), f"sequence {n}: outputs differ"
        assert torch.equal(f1, fin[n:n + 1]), f"sequence {n}: final states differ"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("interval", [32, 64])
def test_checkpoints_equal_prefix_final_states(variant, interval):
    """kda_prefill_checkpointed: outputs and final states are those of
    kda_prefill, and checkpoint j of a sequence is exactly the final state of a
    prefill over its first j * interval tokens (checked bitwise against the
    GPU and within the bound against the oracle)."""
    H, d = 2, 128
    lens = [100, 64, 0, 161]
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(sum(lens), H, d, dtype=dtype, seed=51, device=DEV,
                              num_seqs=len(lens), init_std=0.05)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    try:
        out, fin, ck = kda.kda_prefill_checkpointed(
            inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], init_state=inp["init_state"],
            cu_seqlens=cu, interval=interval, out_dtype=torch.float32, variant=variant)
    except kda.KdaError as e:
        if e.status == 2:
            pytest.skip("variant does not take this shape/dtype (KDA_ERR_UNSUPPORTED)")
        raise
    out0, fin0 = run_gpu(inp, variant, cu=cu)
    assert torch.equal(out, out0) and torch.equal(fin, fin0)
    row = 0
    for n, (t0, t1) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        for j in range(1, (t1 - t0) // interval + 1):
            pre = {x: inp[x][t0:t0 + j * interval].contiguous()
                   for x in ("q", "k", "v", "g", "beta")}
            pre["init_state"] = inp["init_state"][n:n + 1].contiguous()
            _, fin_p = run_gpu(pre, variant)
            assert torch.equal(ck[row], fin_p[0]), f"sequence {n}, checkpoint {j}"
            if j == (t1 - t0) // interval:
                _, s_ref = run_oracle(pre)
                assert rel_err(host64(ck[row]), s_ref[0]) <= TOL[dtype]
            row += 1
    assert row == ck.shape[0]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gated_prefill_matches_oracle(variant, d, dtype):
    """kda_prefill_gated on a ragged packed batch (empty, short, multi-chunk
    sequences) against the oracle fed with the oracle's own gate prologue."""
    if not supported(variant, d, dtype):
        pytest.skip("variant does not take this shape/dtype")
    H = 2
    lens = [1, 31, 32, 0, 65, 100]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=61, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    gl = synth.gate_logits(T, H, d, dtype=dtype, seed=62, device=DEV)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    try:
        out, fin = kda.kda_prefill_gated(inp["q"], inp["k"], inp["v"], gl["z"], gl["a_log"],
                                         gl["beta_logit"], init_state=inp["init_state"],
                                         cu_seqlens=cu, out_dtype=torch.float32, variant=variant)
    except kda.KdaError as e:
        if e.status == 2:
            pytest.skip("variant does not take this shape/dtype (KDA_ERR_UNSUPPORTED)")
        raise
    g, beta = oracle.gate(host64(gl["z"]), host64(gl["a_log"]), host64(gl["beta_logit"]))
    o_ref, s_ref = oracle.prefill(host64(inp["q"]), host64(inp["k"]), host64(inp["v"]), g, beta,
                                  init_state=host64(inp["init_state"]),
                                  cu_seqlens=cu.cpu().numpy())
    check(out, fin, o_ref, s_ref, dtype)


@pytest.mark.parametrize("variant", VARIANTS)
def test_gated_prefill_equals_prefill_of_gate(variant):
    """The fused prologue computes what kda_prefill computes from the same g
    and beta formed outside (oracle gate, rounded to fp32), up to rounding."""
    T, H, d = 150, 2, 128
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=71, device=DEV)
    gl = synth.gate_logits(T, H, d, dtype=dtype, seed=72, device=DEV)
    out, fin = kda.kda_prefill_gated(inp["q"], inp["k"], inp["v"], gl["z"], gl["a_log"],
                                     gl["beta_logit"], out_dtype=torch.float32, variant=variant)
    g, beta = oracle.gate(host64(gl["z"]), host64(gl["a_log"]), host64(gl["beta_logit"]))
    g32 = torch.tensor(g, dtype=torch.float32, device=DEV)
    b32 = torch.tensor(beta, dtype=torch.float32, device=DEV)
    out0, fin0 = kda.kda_prefill(inp["q"], inp["k"], inp["v"], g32, b32,
                                 out_dtype=torch.float32, variant=variant)
    tol = TOL[dtype]
    assert rel_err(host64(out), host64(out0)) <= tol
    assert rel_err(host64(fin), host64(fin0)) <= tol


# ---------------------------------------------------------------------------
# output gate: y = Sigmoid(gate) RMSNorm(o~) w
# ---------------------------------------------------------------------------

OG_EPS = 1e-6


def run_output_gated(inp, og, variant, out_dtype, cu=None, weight=True):
    try:
        return kda.kda_prefill_output_gated(
            inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], og["gate"],
            og["norm_weight"] if weight else None, OG_EPS, init_state=inp.get("init_state"),
            cu_seqlens=cu, out_dtype=out_dtype, variant=variant)
    except kda.KdaError as e:
        if e.status == 2:
            pytest.skip("variant does not take this shape/dtype (KDA_ERR_UNSUPPORTED)")
        raise


def check_bf16_out(out, y_ref, dtype):
    """A bf16 output: the fp32 bound plus half a bf16 ulp of the largest value."""
    ref = np.asarray(y_ref)
    bound = TOL[dtype] + 2.0 ** -8 * np.max(np.abs(ref)) / np.sqrt(np.mean(ref ** 2))
    e = rel_err(host64(out), ref)
    assert e <= bound, f"bf16 output error {e:.3e} > {bound:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_output_gated_matches_oracle(variant, d, dtype, out_dtype):
    """kda_prefill_output_gated on a ragged packed batch against the oracle's
    prefill followed by the oracle's output gate.  A bf16 output on the
    split kernel takes the fused epilogue; the other cases gate in place."""
    if not supported(variant, d, dtype):
        pytest.skip("variant does not take this shape/dtype")
    H = 2
    lens = [1, 31, 32, 0, 65, 100]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=81, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    og = synth.output_gate_inputs(T, H, d, dtype=dtype, seed=82, device=DEV)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    out, fin = run_output_gated(inp, og, variant, out_dtype, cu=cu)
    o_ref, s_ref = run_oracle(inp, cu=cu)
    y_ref = oracle.output_gate(o_ref, host64(og["gate"]), host64(og["norm_weight"]), OG_EPS)
    es = rel_err(host64(fin), s_ref)
    assert es <= TOL[dtype], f"final-state error {es:.3e}"
    if out_dtype == torch.float32:
        eo = rel_err(host64(out), y_ref)
        assert eo <= TOL[dtype], f"gated output error {eo:.3e} > {TOL[dtype]}"
    else:
        check_bf16_out(out, y_ref, dtype)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_output_gate_of_the_kernels_own_readout(variant, out_dtype):
    """The epilogue alone: the gated output equals the gate applied in fp64 to
    the ungated fp32 readout the same kernel writes (kda_prefill), to fp32
    rounding (fp32 out).  A bf16 out is one bf16 rounding away on the fused
    path (the split kernel), and at most two on the in-place path (o~ itself
    goes through bf16 there).  Full chunks and a ragged tail; no weight, then a
    weight."""
    T, H, d = 150, 3, 128
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=91, device=DEV)
    og = synth.output_gate_inputs(T, H, d, dtype=dtype, seed=92, device=DEV)
    o32, _ = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                             out_dtype=torch.float32, variant=variant)
    o = host64(o32)
    gate = host64(og["gate"])
    for weight in (False, True):
        w = host64(og["norm_weight"]) if weight else np.ones(d)
        rinv = 1.0 / np.sqrt((o ** 2).mean(axis=-1, keepdims=True) + OG_EPS)
        y = o * rinv * w / (1.0 + np.exp(-gate))
        out, _ = run_output_gated(inp, og, variant, out_dtype, weight=weight)
        if out_dtype == torch.float32:
            assert np.allclose(host64(out), y, rtol=2e-6, atol=1e-6 * np.abs(y).max())
        else:
            # only the split kernel fuses the gate into its epilogue; every other case
            # gates a bf16 `out` in place after the prefill
            fused = dtype == torch.bfloat16 and variant in (kda.PREFILL_TC_SPLIT, kda.PREFILL_TC_2PASS)
            rel = 2.0 ** -8 if fused else 2.0 ** -7
            assert np.all(np.abs(host64(out) - y) <= rel * np.abs(y) + 1e-6 * np.abs(y).max())


def test_output_gate_zero_rows_stay_zero():
    """Zero values give a zero readout, and the gated output of a zero row is
    zero (eps > 0), on the fused and the in-place paths."""
    T, H, d = 64, 2, 128
    inp = synth.random_inputs(T, H, d, dtype=torch.bfloat16, seed=93, device=DEV)
    inp["v"].zero_()
    og = synth.output_gate_inputs(T, H, d, dtype=torch.bfloat16, seed=94, device=DEV)
    for out_dtype in (torch.float32, torch.bfloat16):
        out, _ = run_output_gated(inp, og, kda.PREFILL_DEFAULT, out_dtype)
        assert torch.count_nonzero(out).item() == 0


# ---------------------------------------------------------------------------
# scalar decay: Gated DeltaNet (one decay per head and step) and the delta rule
# ---------------------------------------------------------------------------

def run_scalar_decay(inp, g_head, variant, out_dtype=torch.float32, cu=None):
    try:
        return kda.kda_prefill_scalar_decay(inp["q"], inp["k"], inp["v"], g_head, inp["beta"],
                                            init_state=inp.get("init_state"), cu_seqlens=cu,
                                            out_dtype=out_dtype, variant=variant)
    except kda.KdaError as e:
        if e.status == 2:
            pytest.skip("variant does not take this shape/dtype (KDA_ERR_UNSUPPORTED)")
        raise


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("decay", ["gated_deltanet", "delta_rule"])
def test_scalar_decay_matches_oracle(variant, d, dtype, decay):
    """kda_prefill_scalar_decay on a ragged packed batch against the oracle's
    scalar-decay recurrence (one decay per head and step, or none)."""
    if not supported(variant, d, dtype):
        pytest.skip("variant does not take this shape/dtype")
    H = 2
    lens = [1, 31, 32, 0, 65, 100]
    T = sum(lens)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=101, device=DEV, num_seqs=len(lens),
                              init_std=0.05)
    gh = synth.scalar_decay(T, H, seed=102, device=DEV) if decay == "gated_deltanet" else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    out, fin = run_scalar_decay(inp, gh, variant, cu=cu)
    o_ref, s_ref = oracle.prefill_scalar_decay(host64(inp["q"]), host64(inp["k"]),
                                               host64(inp["v"]), host64(gh), host64(inp["beta"]),
                                               init_state=host64(inp["init_state"]),
                                               cu_seqlens=cu.cpu().numpy())
    check(out, fin, o_ref, s_ref, dtype)


@pytest.mark.parametrize("variant", VARIANTS)
def test_scalar_decay_equals_prefill_of_broadcast_decay(variant):
    """A scalar decay is the channel-wise decay with one value per head: the
    variant returns exactly (bit for bit) what kda_prefill returns for g
    repeated over the key channels, and the delta rule what it returns for
    g = 0.  Full chunks and a ragged tail, nonzero initial state."""
    T, H, d = 150, 3, 128
    dtype = torch.float32 if supported(variant, d, torch.float32) else torch.bfloat16
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=103, device=DEV, init_std=0.05)
    gh = synth.scalar_decay(T, H, seed=104, device=DEV)
    for g_head, g_full in ((gh, gh[:, :, None].expand(T, H, d).contiguous()),
                           (None, torch.zeros((T, H, d), dtype=torch.float32, device=DEV))):
        out, fin = run_scalar_decay(inp, g_head, variant)
        out0, fin0 = kda.kda_prefill(inp["q"], inp["k"], inp["v"], g_full, inp["beta"],
                                     init_state=inp["init_state"], out_dtype=torch.float32,
                                     variant=variant)
        assert torch.equal(out, out0) and torch.equal(fin, fin0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_output_gate_alone_on_decode_and_gated_outputs(dtype):
    """kda_output_gate in place equals the oracle's gate on the same ungated
    values: on a decode step's output and on kda_prefill_gated's output."""
    T, H, d = 70, 2, 128
    og = synth.output_gate_inputs(T, H, d, dtype=dtype, seed=95, device=DEV)
    inp = synth.random_inputs(T, H, d, dtype=dtype, seed=96, device=DEV)
    gl = synth.gate_logits(T, H, d, dtype=dtype, seed=97, device=DEV)
    o, _ = kda.kda_prefill_gated(inp["q"], inp["k"], inp["v"], gl["z"], gl["a_log"],
                                 gl["beta_logit"], out_dtype=torch.float32)
    ref = oracle.output_gate(host64(o), host64(og["gate"]), host64(og["norm_weight"]), OG_EPS)
    kda.kda_output_gate(o, og["gate"], og["norm_weight"], OG_EPS)
    assert rel_err(host64(o), ref) <= 1e-5
    N = 16
    dec = synth.random_inputs(N, H, d, dtype=dtype, seed=98, device=DEV, num_seqs=N, init_std=0.05)
    state = dec["init_state"].clone()
    od = kda.kda_decode(dec["q"], dec["k"], dec["v"], dec["g"], dec["beta"], state,
                        out_dtype=torch.float32)
    ref = oracle.output_gate(host64(od), host64(og["gate"][:N]), None, OG_EPS)
    kda.kda_output_gate(od, og["gate"][:N].contiguous(), None, OG_EPS)
    assert rel_err(host64(od), ref) <= 1e-5
