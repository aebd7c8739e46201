"""The decode entry point that allocates nothing (forkkv_residual_attn_decode_static).

It is meant for callers that cannot allocate device memory (for instance a
serving engine that gives nearly all free HBM to its own KV-cache pool, or a
plugin host that offers no workspace); its scratch lives in a fixed array of
the library.  Through the C ABI its output must match the regular decode entry
point's within the parity tolerance the other tests use, call after call, even
though every call reuses the array the previous call left behind.  This file
is collected last so that a run stopping at the first failure has already run
every other test.
"""
import pytest
import torch

from disaggregated_kv_attention_gb300 import forkkv as fk
from disaggregated_kv_attention_gb300 import workload as wl
from disaggregated_kv_attention_gb300.paged import params, place
from oracle import residual_attention as ra

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    fk.forkkv_get_device_status()


def _setup(name):
    w = wl.generate(wl.CONFIGS[name])
    P = place(w)
    rope = fk.rope_table(w.cfg.rope_theta, P.max_seq_len)
    ref = torch.full_like(P.q, float("nan"))
    p_ref, keep = params(P, ref, rope=rope)          # regular entry point, caller workspace
    fk.forkkv_residual_attn_decode(p_ref)
    torch.cuda.synchronize()
    return P, rope, ref, keep


def _static_call(P, rope, keep):
    """One call of the entry point that allocates nothing; rope=None makes it build the rotation
    table inside its static array too."""
    out = torch.full_like(P.q, float("nan"))
    info = keep["info"]
    p = fk.attn_params(P.pools, 0, P.q, out, P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len, P.B_k, P.B_v,
                       rope=rope, rope_theta=P.w.cfg.rope_theta, plan=keep["plan"], plan_info=info)
    fk.forkkv_residual_attn_decode_static(p)          # no workspace passed
    torch.cuda.synchronize()
    return out


def _check(out, ref):
    a = out.to(torch.float64).cpu().numpy()
    b = ref.to(torch.float64).cpu().numpy()
    assert ra.within_tolerance(a, b), ra.metrics(a, b)
    assert torch.isfinite(out.float()).all()


def test_static_scratch_decode_matches_regular_decode_on_consecutive_calls():
    big = _setup("llama3_8b_decode")
    small = _setup("tiny_decode")
    for P, rope, ref, keep in (big, small, big):     # calls in a row share the array
        out = _static_call(P, rope, keep)
        _check(out, ref)
        assert fk.forkkv_get_device_status() == 0


def test_static_scratch_builds_the_rotation_table_in_its_array_on_consecutive_calls():
    # rope=None: the entry point builds the rotation table inside the static array as well (after
    # the partials), so consecutive calls of different sizes overwrite each other's table.
    big = _setup("llama3_8b_decode")
    small = _setup("tiny_decode")
    for P, rope, ref, keep in (small, big, small):
        out = _static_call(P, None, keep)
        _check(out, ref)
        assert fk.forkkv_get_device_status() == 0


def test_static_scratch_rejects_workloads_beyond_its_size():
    P, rope, ref, keep = _setup("tiny_decode")
    out = torch.empty_like(P.q)
    info = keep["info"]
    p = fk.attn_params(P.pools, 0, P.q, out, P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len, P.B_k, P.B_v,
                       rope=rope, plan=keep["plan"], plan_info=info)
    p.plan_slots = 1 << 20  # claims more partial slots than the static array can hold
    assert fk.forkkv_decode_workspace_size(p) > fk.STATIC_SCRATCH_BYTES
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_residual_attn_decode_static(p)
    assert e.value.code == fk.ERR_SCRATCH
