"""kda_prefill_noalloc: the prefill for callers that may not allocate device
memory during a call (a host whose caching allocator owns all of the GPU's
memory, a service that keeps allocation off its serving path).  Its scratch
is a fixed array of the library, shared by every call and holding the last
call's contents, so two calls in a row must both give the output of the
ordinary entry point.  This file is collected last: it must pass after the
other tests as well as alone in a fresh process."""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth
from kda_testutil import TOL, rel_err, host64

pytestmark = pytest.mark.gpu


def test_noalloc_matches_kda_prefill_twice_in_a_row():
    dev = "cuda"
    lens = [0, 1, 37, 64, 130, 300]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    inp = synth.random_inputs(sum(lens), 4, 128, dtype=torch.bfloat16, seed=21, device=dev,
                              num_seqs=len(lens), init_std=0.05)
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    # the ordinary entry point running the same kernel with pool scratch
    ref_out, ref_fin = kda.kda_prefill(*args, init_state=inp["init_state"], cu_seqlens=cu,
                                       out_dtype=torch.float32, variant=kda.PREFILL_TC_SPLIT)
    # outputs allocated up front by the caller; the two calls reuse them
    out = torch.empty_like(ref_out)
    fin = torch.empty_like(ref_fin)
    results = []
    for _ in range(2):
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
        kda.kda_prefill_noalloc(*args, init_state=inp["init_state"], cu_seqlens=cu, out=out,
                                final_state=fin, out_dtype=torch.float32)
        torch.cuda.synchronize()
        results.append((out.clone(), fin.clone()))
    assert kda.kda_get_last_device_error() == 0
    for o, f in results:
        assert rel_err(host64(o), host64(ref_out)) <= TOL[torch.bfloat16]
        assert rel_err(host64(f), host64(ref_fin)) <= TOL[torch.bfloat16]
    # the same kernel on the same inputs: the second call repeats the first exactly
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


def test_noalloc_rejects_what_its_array_cannot_hold():
    # d = 64 is not taken by the split kernel: rejected before any launch
    inp = synth.random_inputs(64, 2, 64, dtype=torch.bfloat16, seed=22, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_noalloc(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    assert e.value.status == 2   # KDA_ERR_UNSUPPORTED
