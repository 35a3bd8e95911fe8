"""Bounded device waits in the extend kernel (a test-only limit, rc_debug_set_wait_limit_ns).

Every wait inside the kernel gives up after its limit: the kernel then records code 3 in the
device status word, stops issuing work and returns instead of hanging. Here the limit is cut to
one nanosecond for one call on a small case, so that the kernel's waits run out; the call must
return, the status word must report the expired wait, and the next call with the default limit
must be clean and match the oracle. Nothing faults or hangs: the only failure made is a wait
that stops early.
"""
import numpy as np
import pytest

import synth
from synth import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def test_extend_wait_that_runs_out_reports_and_the_next_call_is_clean():
    import torch
    import prefix_cached_paged_gb300 as rc
    m = W.Model(1, 16, 4, 128, "bf16", 9)
    pre = synth.tokens(9, 1, 300)
    w = W.Workload("wait_limit", m, 8192, synth.permutation(9, 8192), max_ctx=640)
    eng = H.make_engine(w, max_reqs=16, stack_extend=False)
    H.run_cache_phase(eng, m, [pre])
    assert rc.device_status() == 0
    seqs = [np.concatenate([pre, synth.tokens(9, 10 + i, 40 + 70 * i)]).astype(np.int32)
            for i in range(3)]
    rc.set_wait_limit_ns(1)
    try:
        H.run_extend_phase(eng, m, seqs, keep_outputs=False)
        torch.cuda.synchronize()
    finally:
        rc.set_wait_limit_ns(0)
    assert rc.device_status() == 3
    # new suffixes (the failed call's slots hold no valid KV), default limit: clean and correct
    seqs = [np.concatenate([pre, synth.tokens(9, 20 + i, 60 + 50 * i)]).astype(np.int32)
            for i in range(3)]
    b, outs = H.run_extend_phase(eng, m, seqs)
    torch.cuda.synchronize()
    assert rc.device_status() == 0
    for i in range(3):
        for h in range(m.n_kv_heads):
            ref, _ = H.oracle_unit(m, seqs[i], 300, 0, h)
            got = outs[0][0][b.plan.qo_indptr[i]:b.plan.qo_indptr[i + 1], h * 4:h * 4 + 4]
            ok, ma, rl = H.compare(got.float().cpu().numpy(), ref, m.dtype)
            assert ok, (i, h, ma, rl)
