"""Decode parity: the CUDA path through the C-ABI against the fp64 oracle.

Tolerance (stated with the method's target for bf16 inputs and fp32
accumulation): max abs error <= 2e-2 and relative L2 <= 5e-3 over the compared
outputs.  Full-size configurations compare every output the oracle can afford
(all for the 8B- and 7B-shaped workloads, sampled agents and heads for the
70B-shaped tree); the launch configuration is the one bench.py times (plan
built from the page tables, rotation table built once).
"""
import numpy as np
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
    fk.forkkv_get_device_status()


def _run(P, use_plan=True, rope=None, layer=0, target_ctas=0):
    out = torch.full_like(P.q, float("nan"))
    p, keep = params(P, out, layer=layer, use_plan=use_plan, rope=rope, target_ctas=target_ctas)
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    return out


@pytest.mark.parametrize("cfg_name", ["tiny_decode", "llama3_8b_decode", "qwen25_7b_mapreduce_decode"])
def test_decode_parity_full(cfg_name):
    w = wl.generate(wl.CONFIGS[cfg_name])
    P = place(w)
    rope = fk.rope_table(w.cfg.rope_theta, P.max_seq_len)
    out = _run(P, rope=rope)
    ref = oracle(w, range(w.n_agents))
    m, ok = compare(out, ref)
    assert ok, m
    assert torch.isfinite(out.float()).all()


def test_decode_parity_llama3_70b_tree_sampled():
    w = wl.generate(wl.CONFIGS["llama3_70b_stress_decode"])
    P = place(w)
    rope = fk.rope_table(w.cfg.rope_theta, P.max_seq_len)
    out = _run(P, rope=rope)
    G = w.cfg.group
    heads = list(range(0, G)) + list(range(5 * G, 6 * G))   # KV heads 0 and 5
    agents = [0, 17, 38, 63]                                  # one per trunk
    ref = oracle(w, agents, q_heads=heads)
    m, ok = compare(out, ref)
    assert ok, m
    assert torch.isfinite(out.float()).all()


def test_plan_and_no_plan_agree_and_workspace_rope():
    w = wl.generate(wl.CONFIGS["llama3_8b_decode"])
    P = place(w)
    rope = fk.rope_table(w.cfg.rope_theta, P.max_seq_len)
    a = _run(P, use_plan=True, rope=rope)
    b = _run(P, use_plan=False, rope=rope)
    c = _run(P, use_plan=True, rope=None)  # table built inside the workspace
    d = _run(P, use_plan=True, rope=rope, target_ctas=40)
    e = _run(P, use_plan=True, rope=rope)
    assert torch.equal(a, e)  # deterministic
    assert torch.equal(a, c)
    for x in (b, d):
        diff = (x.float() - a.float()).abs().max().item()
        assert diff < 2e-3, diff  # split changes only the fp32 reduction order


def test_sharing_is_invisible():
    # aliased trunk (fork) vs every agent holding a private clone of it
    tree = wl.CONFIGS["tiny_decode"]
    w = wl.generate(tree)
    P_shared = place(w)
    # clone: a flat tree whose agents own all their tokens
    flat_nodes = [wl.Node(f"a{i}", -1, (0, 0), True) for i in range(w.n_agents)]
    cfg_flat = wl.custom_config("flat", tree.n_q_heads, tree.n_kv_heads, flat_nodes, rope_theta=tree.rope_theta)
    wf = wl.Workload(cfg_flat, [int(x) for x in w.seq_lens], [0] * w.n_agents,
                     [w.agent_base(a)[0] for a in range(w.n_agents)], [w.agent_base(a)[1] for a in range(w.n_agents)],
                     w.k_res, w.v_res, w.q, w.B_k, w.B_v, w.seq_lens, w.positions)
    P_clone = place(wf)
    assert len(set(P_shared.bpt_np[:, 0])) == 1 and len(set(P_clone.bpt_np[:, 0])) == w.n_agents
    a = _run(P_shared, use_plan=False)
    b = _run(P_clone, use_plan=False)
    assert torch.equal(a, b)  # same reduction order: bit-identical
    c = _run(P_shared, use_plan=True)
    assert (c.float() - a.float()).abs().max().item() < 2e-3


def _custom(name, Hq, Hkv, nodes, theta=1e6, b_std=0.02, seed=None):
    cfg = wl.custom_config(name, Hq, Hkv, nodes, rope_theta=theta)
    return wl.generate(cfg, seed=seed, b_std=b_std)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (14, 2), (40, 8), (64, 8), (8, 1)])
def test_group_sizes_and_ragged_tails(Hq, Hkv):
    nodes = [wl.Node("root", -1, (700, 700), False)]
    nodes += [wl.Node(f"a{i}", 0, (1, 45), True) for i in range(5)]
    w = _custom(f"g{Hq}_{Hkv}", Hq, Hkv, nodes)
    P = place(w)
    for use_plan in (True, False):
        out = _run(P, use_plan=use_plan, rope=fk.rope_table(w.cfg.rope_theta, P.max_seq_len))
        m, ok = compare(out, oracle(w, range(w.n_agents)))
        assert ok, (use_plan, m)


def test_unaligned_fork_points_and_deep_tree():
    # trunks end mid-page: the children's first private page is a CoW copy of the tail rows
    nodes = [wl.Node("root", -1, (2050, 2050), False), wl.Node("t0", 0, (37, 37), False),
             wl.Node("t1", 0, (3, 3), False), wl.Node("t2", 1, (100, 100), False)]
    nodes += [wl.Node("a0", 1, (5, 5), True), wl.Node("a1", 2, (19, 19), True), wl.Node("a2", 3, (1, 1), True),
              wl.Node("a3", 3, (33, 33), True), wl.Node("a4", 0, (16, 16), True)]
    w = _custom("unaligned", 32, 8, nodes, theta=5e5, b_std=0.2)
    P = place(w)
    assert len(P.jobs) > 0
    for use_plan in (True, False):
        out = _run(P, use_plan=use_plan)
        m, ok = compare(out, oracle(w, range(w.n_agents)))
        assert ok, (use_plan, m)


def test_single_key_returns_first_value():
    nodes = [wl.Node(f"a{i}", -1, (1, 1), True) for i in range(3)]
    w = _custom("single", 16, 4, nodes)
    P = place(w)
    out = _run(P)
    m, ok = compare(out, oracle(w, range(3)))
    assert ok, m


def test_adapter_ids_select_adapters():
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    P = place(w)
    perm = torch.tensor([2, 0, 3, 1], dtype=torch.int32)
    # give the kernel the adapters in a permuted table plus the matching ids
    inv = torch.argsort(perm)
    Bk_perm = P.B_k[inv.long().cuda()].contiguous()  # table[perm[a]] = B[a]
    Bv_perm = P.B_v[inv.long().cuda()].contiguous()
    ids = perm.cuda()
    out = torch.full_like(P.q, float("nan"))
    p, keep = params(P, out)
    p.B_k, p.B_v = Bk_perm.data_ptr(), Bv_perm.data_ptr()
    p.adapter_ids = ids.data_ptr()
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    m, ok = compare(out, oracle(w, range(w.n_agents)))
    assert ok, m


def test_host_validation_rejects_bad_params():
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    P = place(w)
    out = torch.empty_like(P.q)
    p, keep = params(P, out)
    p.head_dim = 64
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_residual_attn_decode(p)
    assert e.value.code == -5
    p, keep = params(P, out)
    p.workspace_bytes = 16
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_residual_attn_decode(p)
    assert e.value.code == -1
    p, keep = params(P, out)
    p.rope_table_positions = 1
    p.rope_table = keep["ws"].data_ptr()
    with pytest.raises(fk.ForkKVError):
        fk.forkkv_residual_attn_decode(p)


def test_bad_device_page_id_is_flagged_not_faulted():
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    P = place(w)
    bpt = P.bpt.clone()
    bpt[1, 3] = P.pools.desc.num_base_pages + 7
    out = torch.empty_like(P.q)
    p = fk.attn_params(P.pools, 0, P.q, out, bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len, P.B_k, P.B_v,
                       rope_theta=w.cfg.rope_theta)
    ws = fk.workspace_for(p)
    fk.forkkv_residual_attn_decode(p)
    st = fk.forkkv_get_device_status()
    assert st & fk.DEV_BAD_PAGE


def test_group_larger_than_eight_is_unsupported():
    nodes = [wl.Node("a0", -1, (20, 20), True)]
    w = _custom("g16", 16, 1, nodes)
    P = place(w)
    out = torch.empty_like(P.q)
    p = fk.attn_params(P.pools, 0, P.q, out, P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len, P.B_k, P.B_v,
                       rope_theta=w.cfg.rope_theta)
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_decode_workspace_size(p)
    assert e.value.code == -5


def test_step_graph_matches_per_layer_calls():
    """One model decode step (new rows written, then attention, for every layer) captured as
    one CUDA graph gives the same bytes as the per-layer calls, again after the inputs'
    contents change between launches; layer 0 matches the oracle."""
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    layers = 3
    dev = torch.device("cuda", 0)
    P = place(w, device=dev, n_layers=layers)
    A = w.cfg.n_agents
    lens = [int(x) for x in w.seq_lens]
    g = torch.Generator().manual_seed(9)
    q_all = torch.stack([P.q.cpu()] + [torch.randn(P.q.shape, generator=g).to(torch.bfloat16)
                                       for _ in range(layers - 1)]).to(dev)
    out_graph = torch.full_like(q_all, float("nan"))
    out_ref = torch.full_like(q_all, float("nan"))
    rows_l = []
    kb = torch.stack([w.agent_base(a)[0][lens[a] - 1] for a in range(A)]).to(dev)
    vb = torch.stack([w.agent_base(a)[1][lens[a] - 1] for a in range(A)]).to(dev)
    kr = torch.stack([w.k_res[a][lens[a] - 1] for a in range(A)]).to(dev)
    vr = torch.stack([w.v_res[a][lens[a] - 1] for a in range(A)]).to(dev)
    sb = torch.tensor([int(P.bpt_np[a, (lens[a] - 1) // 16]) * 16 + (lens[a] - 1) % 16 for a in range(A)],
                      dtype=torch.int32, device=dev)
    sr = torch.tensor([int(P.rpt_np[a, (lens[a] - 1) // 16]) * 16 + (lens[a] - 1) % 16 for a in range(A)],
                      dtype=torch.int32, device=dev)
    for _ in range(layers):
        rows_l.append((sb, sr, kb, vb, kr, vr))
    rope = fk.rope_table(w.cfg.rope_theta, P.max_seq_len, device=dev)
    plan, info = fk.forkkv_plan_build(P.bpt_np, w.seq_lens.numpy(), w.cfg.n_kv_heads)
    plan_d = torch.from_numpy(plan).to(dev)

    def mk(out):
        ps = [fk.attn_params(P.pools, l, q_all[l], out[l], P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len,
                             P.B_k, P.B_v, rope=rope, plan=plan_d, plan_info=info) for l in range(layers)]
        return ps

    p_ref, p_graph = mk(out_ref), mk(out_graph)
    ws = fk.workspace_for(p_ref[0], device=dev)
    for p in p_ref + p_graph:
        fk.set_workspace(p, ws)

    def eager():
        for l in range(layers):
            fk.forkkv_write_rows(P.pools, l, sb, sr, kb, vb, kr, vr)
            fk.forkkv_residual_attn_decode(p_ref[l])

    eager()
    torch.cuda.synchronize()
    graph = fk.forkkv_step_graph_create(p_graph, rows_l)
    try:
        for step in range(2):
            fk.forkkv_step_graph_launch(graph)
            torch.cuda.synchronize()
            assert fk.forkkv_get_device_status() == 0
            assert torch.equal(out_graph.view(torch.int16), out_ref.view(torch.int16)), step
            q_all.mul_(-0.5)  # new contents, same addresses
            eager()
            torch.cuda.synchronize()
    finally:
        fk.forkkv_step_graph_destroy(graph)
    q_all.mul_(1.0 / 0.25)  # back to the layer-0 query of the workload (two halvings, exact in bf16)
    eager()
    torch.cuda.synchronize()
    m, ok = compare(out_ref[0], oracle(w, range(A)))
    assert ok, m


def _stale_plan_run(P, bpt, seq_lens, positions, plan_src):
    """Decode with tables (bpt, seq_lens, positions) but a plan built from plan_src's tables."""
    out = torch.full_like(P.q, float("nan"))
    plan, info = fk.forkkv_plan_build(plan_src[0], plan_src[1], P.w.cfg.n_kv_heads)
    plan_d = torch.from_numpy(plan).to(P.device)
    p = fk.attn_params(P.pools, 0, P.q, out, bpt, P.rpt, seq_lens, positions, P.max_seq_len, P.B_k, P.B_v,
                       rope_theta=P.w.cfg.rope_theta, plan=plan_d, plan_info=info)
    ws = fk.workspace_for(p)
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    del ws
    return fk.forkkv_get_device_status()


def test_stale_plan_after_a_split_page_is_flagged():
    # After a copy-on-write split one agent maps its own copy of a trunk page; a plan built before
    # the split still groups it with the others.  The producer compares every agent's base page
    # ids of a block with the first agent's and reports the mismatch (FORKKV_DEV_BAD_ARG); the
    # kernel still runs to the end.  A plan built from the new tables raises nothing.
    w = wl.generate(wl.CONFIGS["llama3_8b_decode"])
    P = place(w)
    old = (P.bpt_np.copy(), w.seq_lens.numpy().copy())
    bpt = P.bpt.clone()
    bpt[3, 2] = int(P.bpt_np[0, 5])   # agent 3's page 2 now names another (valid) base page
    assert _stale_plan_run(P, bpt, P.seq_lens, P.positions, old) == fk.DEV_BAD_ARG
    assert _stale_plan_run(P, bpt, P.seq_lens, P.positions, (bpt.cpu().numpy(), old[1])) == 0


def test_stale_plan_after_a_sequence_grew_into_a_new_page_is_flagged():
    # An agent whose sequence entered a new page after the plan was built: the plan's items cover
    # fewer pages than its length needs.  The combine kernel checks coverage and reports it.
    w = wl.generate(wl.CONFIGS["llama3_8b_decode"])
    P = place(w)
    old = (P.bpt_np.copy(), w.seq_lens.numpy().copy())
    a = int(np.argmin(old[1]))                       # the shortest agent stays within max_seq_len
    seq_lens, positions = P.seq_lens.clone(), P.positions.clone()
    grow = 16 - (int(old[1][a]) % 16) + 1            # one slot into the page after its last
    seq_lens[a] += grow
    positions[a, 0] += grow
    assert int(seq_lens[a]) <= P.max_seq_len
    bpt = P.bpt.clone()
    new_page = (int(seq_lens[a]) - 1) // 16
    bpt[a, new_page] = int(P.bpt_np[a, 0])
    assert _stale_plan_run(P, bpt, seq_lens, positions, old) & fk.DEV_BAD_ARG
