"""Residual fill and fused decode append on the GPU against the fp64 oracle.

Values: |device - exact| <= half a bf16 unit of the exact value + the fp32
accumulation bound (oracle/residual_fill.py, rounding_bound), and at least 99 %
of the rows' values equal to the oracle's own bf16 rounding.  Placement:
bit-exact (every requested slot holds its row, every other row keeps the fill
pattern).  Shapes: ragged token tiles and a hidden size that is not a multiple
of the 64-element stage; 1 to 8 agents (32 to 256 columns per CTA); the
Llama-3-8B fan-out at full size (8 agents x 8192 prefix tokens, hidden 4096)
on sampled tokens.
"""
import numpy as np
import pytest
import torch

from disaggregated_kv_attention_gb300 import forkkv as fk
from gpu_harness import base_tile_rows, res_tile_rows
from oracle.residual_fill import bf16_round, residual_rows, rounding_bound

pytestmark = pytest.mark.gpu
FILL = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    assert fk.forkkv_get_device_status() == 0


def _bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _res_rows_all(tiles: np.ndarray) -> np.ndarray:
    """[n_pages][512] uint8 residual tiles -> [n_pages * 16][16] uint16 rows (logical order), the layout
    of include/forkkv.h (32-byte rows, 16-byte halves swapped on rows 4..7 and 12..15)."""
    t = np.arange(16)[:, None]
    k = np.arange(16)[None, :]
    idx = (t * 32 + (((k // 8) ^ ((t // 4) % 2)) * 16) + (k % 8) * 2) // 2
    return tiles.view(np.uint16)[:, idx].reshape(-1, 16)


def _inputs(seed, n_tok, hidden, n_ag):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n_tok, hidden, generator=g).to(torch.bfloat16)
    A = (0.02 * torch.randn(n_ag, 2, 16, hidden, generator=g)).to(torch.bfloat16)
    return x, A


def _check_rows(got_k, got_v, x, A, agent_idx, tok_idx):
    """got_k/v [n][16] bf16 bits of the (agent_idx[i], tok_idx[i]) pairs."""
    xs = x.to(torch.float64).numpy()
    Ad = A.to(torch.float64).numpy()
    got = np.stack([_bf16_bits_to_f64(got_k), _bf16_bits_to_f64(got_v)], axis=1)  # [n][2][16]
    agent_idx, tok_idx = np.asarray(agent_idx), np.asarray(tok_idx)
    same = 0
    for a in np.unique(agent_idx):
        sel = np.nonzero(agent_idx == a)[0]
        xt = xs[tok_idx[sel]]
        exact = residual_rows(xt, Ad[a:a + 1])[0]            # [n_a][2][16]
        bound = rounding_bound(xt, Ad[a:a + 1], exact[None])[0]
        err = np.abs(got[sel] - exact)
        assert np.all(err <= bound), (int(a), float((err - bound).max()))
        same += int(np.sum(got[sel] == bf16_round(exact)))
    frac = same / got.size
    assert frac >= 0.99, frac


# the last two shapes give 153 token tiles, so that 8 and 5 agents share one CTA (256 and 160 columns)
@pytest.mark.parametrize("n_tok,hidden,n_ag", [(300, 520, 3), (129, 64, 1), (64, 256, 8), (1000, 1024, 5),
                                               (19500, 512, 8), (19500, 264, 5)])
def test_residual_fill_small(n_tok, hidden, n_ag):
    n_res = (n_ag * n_tok + 15) // 16 + 4
    pools = fk.Pools(8, n_res, 2, n_layers=2, fill=FILL)
    x, A = _inputs(n_tok + hidden + n_ag, n_tok, hidden, n_ag)
    g = torch.Generator().manual_seed(7)
    slots = torch.randperm(n_res * 16, generator=g)[:n_ag * n_tok].to(torch.int32).view(n_ag, n_tok)
    skip = torch.rand(n_ag, n_tok, generator=g) < 0.05
    slots[skip] = -1
    fk.forkkv_residual_fill(pools, 1, x.cuda(), A.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    kr = pools.k_res.cpu().numpy()
    vr = pools.v_res.cpu().numpy()
    assert np.all(kr[0] == FILL) and np.all(vr[0] == FILL)  # the other layer is untouched
    rows_k, rows_v = _res_rows_all(kr[1]), _res_rows_all(vr[1])
    assert np.array_equal(rows_k[:16], res_tile_rows(kr[1, 0]))  # the fast decoder agrees with the harness
    s = slots.numpy()
    written = s[s >= 0]
    untouched = np.setdiff1d(np.arange(n_res * 16), written)
    fill16 = np.uint16(FILL | (FILL << 8))
    assert np.all(rows_k[untouched] == fill16) and np.all(rows_v[untouched] == fill16)
    agent_idx, tok_idx = np.nonzero(s >= 0)
    sl = s[agent_idx, tok_idx]
    _check_rows(rows_k[sl], rows_v[sl], x, A, agent_idx, tok_idx)


def test_residual_fill_full_size_fanout():
    """Eight agents forked from an 8192-token prefix of a Llama-3-8B-shaped model (hidden 4096):
    every agent's residual rows of every prefix token in one call; sampled tokens checked."""
    n_tok, hidden, n_ag = 8192, 4096, 8
    n_res = n_ag * n_tok // 16
    pools = fk.Pools(8, n_res, 8, n_layers=1, fill=FILL)
    x, A = _inputs(88, n_tok, hidden, n_ag)
    # each agent's prefix in its own run of residual pages, agents interleaved page by page
    t = torch.arange(n_tok)
    slots = torch.stack([((t // 16) * n_ag + a) * 16 + t % 16 for a in range(n_ag)]).to(torch.int32)
    fk.forkkv_residual_fill(pools, 0, x.cuda(), A.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    rng = np.random.default_rng(0)
    toks = np.concatenate([rng.choice(n_tok, 120, replace=False), [0, 127, 128, n_tok - 1]])
    kr = pools.k_res[0].cpu().numpy()
    vr = pools.v_res[0].cpu().numpy()
    agent_idx = np.repeat(np.arange(n_ag), len(toks))
    tok_idx = np.tile(toks, n_ag)
    sl = slots.numpy()[agent_idx, tok_idx]
    rows_k, rows_v = _res_rows_all(kr), _res_rows_all(vr)
    _check_rows(rows_k[sl], rows_v[sl], x, A, agent_idx, tok_idx)
    assert not np.any(rows_k == np.uint16(FILL | (FILL << 8)))  # every slot was written


def test_append_rows_fused():
    n, hidden, hkv, n_ad = 8, 4096, 8, 6
    pools = fk.Pools(16, 16, hkv, n_layers=2, fill=FILL)
    g = torch.Generator().manual_seed(12)
    x = torch.randn(n, hidden, generator=g).to(torch.bfloat16)
    A = (0.02 * torch.randn(n_ad, 2, 16, hidden, generator=g)).to(torch.bfloat16)
    ids = torch.tensor([3, 0, 5, 5, 1, 2, 4, 0], dtype=torch.int32)
    kb = torch.randn(n, hkv, 128, generator=g).to(torch.bfloat16)
    vb = torch.randn(n, hkv, 128, generator=g).to(torch.bfloat16)
    sb = torch.randperm(16 * 16, generator=g)[:n].to(torch.int32)
    sr = torch.randperm(16 * 16, generator=g)[:n].to(torch.int32)
    sr[6] = -1  # row 6 writes no residual row
    fk.forkkv_append_rows(pools, 1, sb.cuda(), sr.cuda(), kb.cuda(), vb.cuda(), x.cuda(), A.cuda(), ids.cuda())
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    kbase = pools.k_base[1].cpu().numpy()
    vbase = pools.v_base[1].cpu().numpy()
    for i in range(n):
        p, r = int(sb[i]) // 16, int(sb[i]) % 16
        for h in range(hkv):
            assert np.array_equal(base_tile_rows(kbase[h, p])[r], kb[i, h].view(torch.int16).numpy().view(np.uint16))
            assert np.array_equal(base_tile_rows(vbase[h, p])[r], vb[i, h].view(torch.int16).numpy().view(np.uint16))
    kr = pools.k_res[1].cpu().numpy()
    vr = pools.v_res[1].cpu().numpy()
    rows = [i for i in range(n) if sr[i] >= 0]
    got_k = np.stack([res_tile_rows(kr[int(sr[i]) // 16])[int(sr[i]) % 16] for i in rows])
    got_v = np.stack([res_tile_rows(vr[int(sr[i]) // 16])[int(sr[i]) % 16] for i in rows])
    # the oracle works per (adapter, token): give each row its own token index into x
    _check_rows(got_k, got_v, x, A, ids.numpy()[rows], np.array(rows))
    # every other residual row keeps the fill pattern
    written = {int(sr[i]) for i in rows}
    fill16 = np.uint16(FILL | (FILL << 8))
    for s in range(16 * 16):
        if s not in written:
            assert np.all(res_tile_rows(kr[s // 16])[s % 16] == fill16)
            assert np.all(res_tile_rows(vr[s // 16])[s % 16] == fill16)
