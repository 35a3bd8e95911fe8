"""The decode entry point that allocates nothing (rc_decode_attention_noalloc).

Callers such as plugin interfaces that receive only input and output buffers, or serving loops
that forbid device allocation once running, cannot hand the library a workspace. This variant
keeps its split-K scratch in a fixed area inside the library; here it must give the same
outputs as the workspace entry point, on two calls in a row (the area keeps the previous call's
contents, so the second call checks that nothing stale leaks in), and reject arguments whose
scratch would not fit. This file sorts last so that a stop-at-first-failure run has already run
everything else.
"""
import numpy as np
import pytest

import synth
from synth import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def _setup():
    import torch
    m = W.Model(1, 32, 8, 128, "bf16", 21)
    L = [1, 40, 513, 1024, 2500, 4100, 97]
    seqs = [synth.tokens(21, 70 + i, n) for i, n in enumerate(L)]
    w = W.Workload("noalloc", m, 12_000, synth.permutation(21, 12_000), max_ctx=4112)
    eng = H.make_engine(w, max_reqs=16, kv_chunk=256)
    H.run_cache_phase(eng, m, [s[:-1] for s in seqs if len(s) > 1])
    db = eng.decode_begin([s[:-1] for s in seqs])
    eng.decode_step(db)
    h = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in seqs], dtype=np.uint64)
    from synth import device as sdev
    q, k, v = H.dense_qkv(m, sdev.hashes_to_device(h), 0, len(seqs))
    return m, eng, db, q, k, v, seqs


def _call_noalloc(eng, db, q, k, v, o, lse, chunk, mt):
    import prefix_cached_paged_gb300 as rc
    rc.decode_attention_noalloc(q, k, v, db.dev_out_loc, db.dev_seq_len, db.dev_req_idx,
                                eng.dev.req_to_token, eng.dev.k[0], eng.dev.v[0], o,
                                sm_scale=eng.sm_scale, max_total_tokens=mt, kv_chunk=chunk,
                                lse=lse)


def test_noalloc_decode_matches_workspace_decode_twice():
    """Same kernels, same job list, same inputs: the outputs must be bit-identical to the
    workspace entry point's, on two calls in a row and again after a call with another batch
    shape has left its own job list and partial states in the shared area."""
    import torch
    import prefix_cached_paged_gb300 as rc
    m, eng, db, q, k, v, seqs = _setup()
    mt = int(db.seq_len.sum())
    o_ref = torch.empty_like(q)
    l_ref = torch.empty((len(seqs), m.n_q_heads), dtype=torch.float32, device="cuda")
    eng.decode_layer(db, 0, q, k, v, o_ref, lse=l_ref, max_total_tokens=mt)

    def checked_call(tag):
        o = torch.full_like(q, float("nan"))
        l = torch.full_like(l_ref, float("nan"))
        _call_noalloc(eng, db, q, k, v, o, l, 256, mt)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), tag
        assert torch.equal(l, l_ref), tag
        return o

    checked_call("first call")
    checked_call("second call in a row")
    # another shape in between: the first three requests only, 128-token chunks
    n = 3
    o3 = torch.full_like(q[:n], float("nan"))
    rc.decode_attention_noalloc(q[:n], k[:n], v[:n], db.dev_out_loc[:n], db.dev_seq_len[:n],
                                db.dev_req_idx[:n], eng.dev.req_to_token, eng.dev.k[0],
                                eng.dev.v[0], o3, sm_scale=eng.sm_scale,
                                max_total_tokens=int(db.seq_len[:n].sum()), kv_chunk=128)
    torch.cuda.synchronize()
    ok, ma, rl = H.compare(o3.float().cpu().numpy(), o_ref[:n].float().cpu().numpy(), m.dtype)
    assert ok, ("other shape", ma, rl)
    o = checked_call("after a call with another shape")
    # and against the oracle for a few units
    for b in (0, 3, 5):
        ref, _ = H.oracle_unit(m, seqs[b], len(seqs[b]) - 1, 0, 2)
        got = o[b, 2 * m.group:3 * m.group].float().cpu().numpy()[None]
        assert H.compare(got, ref, m.dtype)[0]
    assert rc.device_status() == 0


def test_noalloc_rejects_arguments_beyond_its_scratch():
    import torch
    import prefix_cached_paged_gb300 as rc
    m, eng, db, q, k, v, seqs = _setup()
    o = torch.empty_like(q)
    # an upper bound of 10^9 context tokens at 64-token chunks needs far more than the area
    with pytest.raises(rc.RcError) as e:
        _call_noalloc(eng, db, q, k, v, o, None, 64, 10**9)
    assert e.value.code == rc.RC_ERR_INVALID
    assert "scratch" in str(e.value)
