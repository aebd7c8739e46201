"""Failure detection on the GPU without a GPU fault: a bounded device wait that
runs out reports FORKKV_DEV_TIMEOUT through the device status word, and the
context stays usable (a decode right after it is correct and sets no bit).

The wait that runs out is the self-test's: one thread waits, through the same
routine as every pipeline wait in the kernels, on an mbarrier that nothing
completes, with a short poll limit."""
import pytest
import torch

from disaggregated_kv_attention_gb300 import forkkv as fk
from disaggregated_kv_attention_gb300 import workload as wl
from gpu_harness import compare, oracle, params, place

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    fk.forkkv_get_device_status()  # start from a clear status word


def test_bounded_wait_runs_out_and_reports_timeout():
    for polls in (1, 64, 4096):
        fk.forkkv_wait_selftest(polls)
        st = fk.forkkv_get_device_status()
        assert st == fk.DEV_TIMEOUT, (polls, st)
    assert fk.forkkv_get_device_status() == 0  # reading cleared it


def test_context_usable_after_a_timeout():
    fk.forkkv_wait_selftest(16)
    assert fk.forkkv_get_device_status() == fk.DEV_TIMEOUT
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    P = place(w)
    out = torch.full_like(P.q, float("nan"))
    p, keep = params(P, out, rope=fk.rope_table(w.cfg.rope_theta, P.max_seq_len))
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    m, ok = compare(out, oracle(w, range(w.n_agents)))
    assert ok, m
