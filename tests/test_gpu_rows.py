"""GPU checks of the byte-moving kernels: bit-exact row scatter and copy-on-write
row copies (rows >= n_valid untouched), the rotation table, and the device
status word fed by the kernels' own bounds checks."""
import math

import numpy as np
import pytest
import torch

from disaggregated_kv_attention_gb300 import forkkv as fk
from gpu_harness import base_tile_rows, res_tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    assert fk.forkkv_get_device_status() == 0


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def test_write_rows_bit_exact():
    g = torch.Generator().manual_seed(1)
    Hkv, n_pages, n = 4, 10, 70
    pools = fk.Pools(n_pages, n_pages, Hkv, n_layers=2, fill=0x5A)
    slots = torch.randperm(n_pages * 16, generator=g)[:n].to(torch.int32)
    rslots = torch.randperm(n_pages * 16, generator=g)[:n].to(torch.int32)
    kb = torch.randn(n, Hkv, 128, generator=g).to(torch.bfloat16)
    vb = torch.randn(n, Hkv, 128, generator=g).to(torch.bfloat16)
    kr = torch.randn(n, 16, generator=g).to(torch.bfloat16)
    vr = torch.randn(n, 16, generator=g).to(torch.bfloat16)
    fk.forkkv_write_rows(pools, 1, slots.cuda(), rslots.cuda(), kb.cuda(), vb.cuda(), kr.cuda(), vr.cuda())
    torch.cuda.synchronize()
    kbase = pools.k_base[1].cpu().numpy()
    vbase = pools.v_base[1].cpu().numpy()
    kres = pools.k_res[1].cpu().numpy()
    vres = pools.v_res[1].cpu().numpy()
    for i in range(n):
        pg, t = divmod(int(slots[i]), 16)
        for h in range(Hkv):
            assert np.array_equal(base_tile_rows(kbase[h, pg])[t], _bits(kb[i, h]))
            assert np.array_equal(base_tile_rows(vbase[h, pg])[t], _bits(vb[i, h]))
        pg, t = divmod(int(rslots[i]), 16)
        assert np.array_equal(res_tile_rows(kres[pg])[t], _bits(kr[i]))
        assert np.array_equal(res_tile_rows(vres[pg])[t], _bits(vr[i]))
    # layer 0 untouched
    assert (pools.k_base[0] == 0x5A).all() and (pools.v_res[0] == 0x5A).all()


@pytest.mark.parametrize("share_res", [False, True])
def test_fork_unaligned_tail_copies_valid_rows_only(share_res):
    # ForkServe "unaligned_pack": a 2050-token trunk forked by 4 children
    L, k, Hkv, layers = 2050, 4, 2, 3
    alloc = fk.forkkv_alloc_create(200, 700)  # children get fresh residual pages for the prefix
    pools = fk.Pools(200, 700, Hkv, n_layers=layers, fill=0)
    g = torch.Generator().manual_seed(2)
    for t in (pools.k_base, pools.v_base, pools.k_res, pools.v_res):
        t.copy_(torch.randint(0, 256, t.shape, generator=g, dtype=torch.uint8))
    before = [t.clone() for t in (pools.k_base, pools.v_base, pools.k_res, pools.v_res)]
    root = fk.forkkv_seq_create(alloc, L)
    jobs = []
    for _ in range(k):
        c, j = fk.forkkv_fork(alloc, root, L, fk.FORK_SHARE_RES if share_res else 0)
        jobs += j
    assert len(jobs) == k * (2 if share_res else 1)
    fk.forkkv_cow_copy_rows(pools, jobs)
    torch.cuda.synchronize()
    after = [t.cpu().numpy() for t in (pools.k_base, pools.v_base, pools.k_res, pools.v_res)]
    before = [t.cpu().numpy() for t in before]
    touched_base = {j[1] for j in jobs if j[3] == fk.JOB_BASE}
    touched_res = {j[1] for j in jobs if j[3] == fk.JOB_RES}
    for src, dst, nv, kind in jobs:
        assert nv == L % 16
        for layer in range(layers):
            if kind == fk.JOB_BASE:
                for pool in (0, 1):
                    for h in range(Hkv):
                        s_rows = base_tile_rows(before[pool][layer, h, src])
                        d_before = base_tile_rows(before[pool][layer, h, dst])
                        d_after = base_tile_rows(after[pool][layer, h, dst])
                        assert np.array_equal(d_after[:nv], s_rows[:nv])
                        assert np.array_equal(d_after[nv:], d_before[nv:])
            else:
                for pool in (2, 3):
                    s_rows = res_tile_rows(before[pool][layer, src])
                    d_after = res_tile_rows(after[pool][layer, dst])
                    assert np.array_equal(d_after[:nv], s_rows[:nv])
                    assert np.array_equal(d_after[nv:], res_tile_rows(before[pool][layer, dst])[nv:])
    # no other page changed
    for pool, touched, axis in ((0, touched_base, 2), (1, touched_base, 2), (2, touched_res, 1),
                                (3, touched_res, 1)):
        mask = np.ones(after[pool].shape[axis], bool)
        mask[list(touched)] = False
        assert np.array_equal(np.compress(mask, after[pool], axis), np.compress(mask, before[pool], axis))
    fk.forkkv_alloc_destroy(alloc)


def test_cow_copy_rejects_bad_jobs_on_host():
    pools = fk.Pools(4, 4, 1)
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_cow_copy_rows(pools, [(0, 4, 3, fk.JOB_BASE)])
    assert e.value.code == -3
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_cow_copy_rows(pools, [(0, 1, 17, fk.JOB_BASE)])
    assert e.value.code == -1


def test_many_cow_jobs_batch_over_launches():
    n_pages, Hkv = 700, 1
    pools = fk.Pools(n_pages, n_pages, Hkv, fill=0)
    pools.k_base.copy_(torch.randint(0, 256, pools.k_base.shape, dtype=torch.uint8))
    jobs = [(i, 350 + i, 16, fk.JOB_BASE) for i in range(300)]  # spans two launches
    fk.forkkv_cow_copy_rows(pools, jobs)
    torch.cuda.synchronize()
    assert torch.equal(pools.k_base[0, 0, 350:650], pools.k_base[0, 0, 0:300])


def test_rope_table_matches_float64_trig():
    theta = 500000.0
    n = 2 ** 17 + 64
    t = fk.rope_table(theta, n)
    torch.cuda.synchronize()
    raw = t.cpu().numpy().reshape(-1)
    pos = np.array([0, 1, 2, 15, 16, 1000, 65535, 2 ** 17, 2 ** 17 + 17, n - 1])
    f = theta ** (-np.arange(0, 128, 2, dtype=np.float64) / 128)
    for p in pos:
        for m in range(32):
            off = (p >> 4) * 4096 + (m >> 2) * 512 + (p & 15) * 32 + (m & 3) * 8  # page-major layout
            bits = raw[off:off + 8].view(np.uint16).astype(np.uint32) << 16
            vals = bits.view(np.float32).astype(np.float64)  # bf16 -> fp32 is exact
            ang = p * f[2 * m:2 * m + 2]
            assert np.allclose(vals[:2], np.cos(ang), atol=4e-3, rtol=0), (p, m)  # bf16: 2^-9 relative
            assert np.allclose(vals[2:], np.sin(ang), atol=4e-3, rtol=0), (p, m)


def test_device_status_records_out_of_range_slot():
    pools = fk.Pools(2, 2, 1)
    bad = torch.tensor([5 * 16], dtype=torch.int32, device="cuda")  # page 5 of a 2-page pool
    kb = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device="cuda")
    fk.forkkv_write_rows(pools, 0, bad, None, kb, kb, None, None)
    st = fk.forkkv_get_device_status()
    assert st & fk.DEV_BAD_PAGE
    assert fk.forkkv_get_device_status() == 0  # read clears
