"""Plan-time memory model and job sharding (host only, no GPU)."""
import numpy as np
import pytest

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from adapter_gemm_packed_gb300.layer import host_plan


@pytest.fixture(scope="module", autouse=True)
def built():
    from adapter_gemm_packed_gb300 import build
    build.build()


def test_memory_estimate_hand_worked():
    # d_in=64, d_out=32, ranks {2,3}, tokens {5,7}, bf16 activations
    plan, ws = host_plan(64, 32, [2, 3], [5, 7])
    try:
        m = M.mlora_memory_estimate(plan)
    finally:
        M.mlora_plan_destroy(plan)
    assert m["base_weight"] == 64 * 32 * 2
    assert m["activations"] == 12 * (64 + 32) * 2 * 2          # X, dX and Y, dY
    assert m["lora_params"] == (2 + 3) * (64 + 32) * 4            # fp32 masters
    assert m["lora_grad_state"] == 3 * (2 + 3) * (64 + 32) * 4    # gradient, first and second moment
    assert m["lora_act"] == (5 * 2 + 7 * 3) * 4 * 2               # H and dH
    assert m["workspace"] == ws
    assert m["total"] == sum(v for k, v in m.items() if k != "total")


def test_memory_estimate_matches_paper_terms_per_job():
    """PLoRA §8 per job k: M_param = (h_in r + h_out r) c_prec, M_grad = c_grad M_param with c_grad = 3,
    M_act = b s r c_prec; summed over jobs they give the library's adapter terms (c_prec = 4)."""
    wl = W.mlp_up_lognormal()
    plan, _ = host_plan(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens)
    try:
        m = M.mlora_memory_estimate(plan)
    finally:
        M.mlora_plan_destroy(plan)
    c_prec, c_grad = 4, 3
    params = sum((wl.d_in * r + wl.d_out * r) * c_prec for r in wl.ranks)
    act = sum(n * r * c_prec for n, r in zip(wl.n_tokens, wl.ranks))
    assert m["lora_params"] == params
    assert m["lora_grad_state"] == c_grad * params
    assert m["lora_act"] == 2 * act


def _segs(ns, rs):
    out, off = [], 0
    for i, (n, r) in enumerate(zip(ns, rs)):
        out.append(M.mlora_segment(off, n, r, 1.0, 0x1000, 0x2000, 0, 0, 0, 0, 0, 0))
        off += n
    return out


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 8])
def test_shard_jobs_assigns_every_job_and_balances(n_ranks):
    wl = W.llama70b_down_many_small()
    prob = M.mlora_problem(wl.N, wl.d_in, wl.d_out, M.MLORA_BF16, M.MLORA_PLAN_HOST_ONLY)
    ranks, load = M.mlora_shard_jobs(prob, _segs(wl.n_tokens, wl.ranks), n_ranks)
    assert len(ranks) == wl.n_adapters and all(0 <= r < n_ranks for r in ranks)
    cost = [n * (wl.d_in * wl.d_out + 3 * r * (wl.d_in + wl.d_out)) for n, r in zip(wl.n_tokens, wl.ranks)]
    per = np.zeros(n_ranks)
    for c, r in zip(cost, ranks):
        per[r] += c
    assert np.allclose(per, load)
    assert per.sum() == pytest.approx(sum(cost))
    # longest-processing-time-first: the spread is at most the largest single job
    assert per.max() - per.min() <= max(cost) + 1e-6 * per.max()


def test_shard_jobs_rejects_bad_input():
    prob = M.mlora_problem(10, 64, 64, M.MLORA_BF16, 0)
    with pytest.raises(M.MloraError):
        M.mlora_shard_jobs(prob, _segs([10], [4]), 0)


def test_plan_refuses_a_pack_over_its_memory_budget():
    """PLoRA §8's constraint as a plan-time check: a budget below the estimate's total is refused
    with MLORA_ERR_OOM, the exact total is accepted, and 0 means no check."""
    plan, _ = host_plan(64, 32, [2, 3], [5, 7])
    try:
        total = M.mlora_memory_estimate(plan)["total"]
    finally:
        M.mlora_plan_destroy(plan)
    with pytest.raises(M.MloraError) as e:
        host_plan(64, 32, [2, 3], [5, 7], mem_budget=total - 1)
    assert e.value.status == M.MLORA_ERR_OOM and str(total) in str(e.value)
    for budget in (total, 0):
        plan, _ = host_plan(64, 32, [2, 3], [5, 7], mem_budget=budget)
        M.mlora_plan_destroy(plan)


def test_cost_estimate_hand_worked():
    """Step time from a table of measured steps (PLoRA §3.1-§3.2's T(H, 1)), worked by hand.
    The plan: d_in = 64, d_out = 32, ranks {2, 3}, tokens {5, 7}: N = 12 and the adapters' work
    5*2*(64+32) + 7*3*(64+32) = 2976, so F = 4*12*64*32 + 6*2976 = 98304 + 17856 = 116160."""
    plan, _ = host_plan(64, 32, [2, 3], [5, 7])
    try:
        # two points of this shape: F = 4*6*2048 + 6*1000 = 55152 (1 ms) and 4*24*2048 + 6*4000 = 220608 (3 ms);
        # a point of another shape that must not be used while this shape has points
        pts = [(64, 32, 6, 1000.0, 1.0), (64, 32, 24, 4000.0, 3.0), (128, 128, 12, 0.0, 0.01)]
        ms, basis = M.mlora_cost_estimate(plan, pts)
        assert basis == 0 and ms == pytest.approx(1.0 + (116160 - 55152) * (3.0 - 1.0) / (220608 - 55152))
        # above the largest point: F at that point's rate, 116160 / (55152 / 1 ms)
        ms, basis = M.mlora_cost_estimate(plan, pts[:1])
        assert basis == 1 and ms == pytest.approx(116160 / 55152)
        # no point of this shape: the rate of the point nearest in work, F = 4*12*128*128 = 786432 in 0.01 ms
        ms, basis = M.mlora_cost_estimate(plan, pts[2:])
        assert basis == 2 and ms == pytest.approx(116160 / (786432 / 0.01))
        with pytest.raises(M.MloraError):
            M.mlora_cost_estimate(plan, [(64, 32, 6, 1000.0, 0.0)])
    finally:
        M.mlora_plan_destroy(plan)


def test_shipped_cost_table_covers_the_layer_shapes():
    """The table measured on a GB300 (adapter_gemm_packed_gb300/cost_table_gb300.json) has points
    for every projection of the Llama-3-8B layer, and its estimate for the layer's own q projection
    lies within the measured points' rates."""
    from adapter_gemm_packed_gb300 import cost
    table = cost.load_table()
    shapes = {(p[0], p[1]) for p in table}
    for _, din, dout in W.LLAMA8B_PROJ:
        assert (din, dout) in shapes
    wl = W.llama8b_layer(0)
    plan, _ = host_plan(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens)
    try:
        ms, basis = M.mlora_cost_estimate(plan, table)
    finally:
        M.mlora_plan_destroy(plan)
    assert basis in (0, 1) and ms > 0
    rates = [(4.0 * n * a * b + 6.0 * w) / t for a, b, n, w, t in table if (a, b) == (wl.d_in, wl.d_out)]
    f = 4.0 * wl.N * wl.d_in * wl.d_out + 6.0 * sum(n * r * (wl.d_in + wl.d_out) for n, r in zip(wl.n_tokens, wl.ranks))
    assert min(rates) * 0.999 <= f / ms <= max(rates) * 1.001
