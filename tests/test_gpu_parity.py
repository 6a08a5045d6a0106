"""CUDA path vs the fp64 oracle, element by element, through the C ABI (needs a GB300).

Small and medium cases run the whole oracle; they span several 128-token tiles, ragged token
and column tails, ranks 1..256 and jobs that straddle tiles."""
import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from oracle import lora_oracle as orc
import gpu_harness as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adapter_gemm_packed_gb300 import build
    build.build()


def _run(wl, keys=None, **kw):
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, **kw)
    try:
        assert run.status_after_backward == M.MLORA_OK
        want = G.oracle_full(wl, T, kw.get("Wt_override"))
        return G.compare(run.res, want, G.TOL[wl.dtype], keys), run.res, want
    finally:
        run.close()


def test_tiny_f32_all_outputs():
    errs, _, _ = _run(W.tiny_f32())
    assert errs["Y"] < 1e-5


F32_CASES = {
    "ragged": dict(d_in=200, d_out=136, ranks=[1, 7, 64, 256], n_tokens=[70, 1, 129, 33]),
    "tiles": dict(d_in=512, d_out=384, ranks=[16, 32, 3], n_tokens=[300, 64, 513]),
    "one_job_rank256": dict(d_in=256, d_out=320, ranks=[256], n_tokens=[200]),
    # enough 128 x 128 tiles (33 x 11) for the large-tile base products in both directions
    "large_tiles": dict(d_in=1292, d_out=1288, ranks=[16, 200, 1, 64], n_tokens=[1500, 1100, 37, 1500]),
}


@pytest.mark.parametrize("name", sorted(F32_CASES))
def test_f32_cases(name):
    """The fp32 path beyond the tiny workload: several 64 x 64 tiles, ragged rows and columns, a
    one-token job, jobs straddling row tiles, ranks 1 to 256 (true fp32 arithmetic, 1e-4)."""
    cfg = F32_CASES[name]
    wl = W.custom(f"f32_{name}", 940 + sorted(F32_CASES).index(name), cfg["d_in"], cfg["d_out"], cfg["ranks"],
                  cfg["n_tokens"], dtype="f32", w_std=0.05, b_std=0.05)
    _run(wl)


SMALL_BF16 = {
    "ragged_tail": dict(d_in=512, d_out=640, ranks=[1, 7, 64, 256], n_tokens=[200, 56, 300, 17]),
    "jobs_straddle_tiles": dict(d_in=256, d_out=384, ranks=[1, 2, 4, 8, 16, 32, 64, 128, 256, 3],
                                n_tokens=[16, 16, 32, 16, 48, 16, 16, 64, 16, 5]),
    "single_token_job": dict(d_in=128, d_out=136, ranks=[5], n_tokens=[1]),
    "one_job_many_tiles": dict(d_in=1024, d_out=512, ranks=[32], n_tokens=[1000]),
    "wide_hidden": dict(d_in=2048, d_out=1536, ranks=[16, 128, 8], n_tokens=[256, 384, 130]),
    # d_in and d_out not multiples of 64: the base GEMMs' TMA stores clip a partial 64-column box
    "ragged_columns": dict(d_in=264, d_out=200, ranks=[8, 33, 128], n_tokens=[300, 45, 170]),
}


ENGINES = {"cta_pairs": 0, "single_cta": M.MLORA_GEMM_SINGLE_CTA}
# the shrink / dH products: on CTA pairs (256-token tiles, up to 4 chunks) or single CTAs
WINDOWS = {"win_pairs": M.MLORA_WINDOW_PAIRS, "win_single": M.MLORA_WINDOW_SINGLE}


@pytest.mark.parametrize("window", sorted(WINDOWS))
@pytest.mark.parametrize("engine", sorted(ENGINES))
@pytest.mark.parametrize("name", sorted(SMALL_BF16))
def test_bf16_small(name, engine, window):
    cfg = SMALL_BF16[name]
    wl = W.custom(f"small_{name}", 900 + sorted(SMALL_BF16).index(name), cfg["d_in"], cfg["d_out"], cfg["ranks"],
                  cfg["n_tokens"], dtype="bf16", w_std=0.05, b_std=0.05)
    _run(wl, flags=ENGINES[engine] | WINDOWS[window])


def test_bf16_zero_base_weight_isolates_rank_term():
    wl = W.custom("zero_W", 950, 512, 384, [4, 64, 17], [130, 200, 70], dtype="bf16", b_std=0.05)
    zero = np.zeros((wl.d_out, wl.d_in), np.uint16)
    errs, got, want = _run(wl, Wt_override=zero)
    assert np.linalg.norm(want["Y"]) > 0


def test_bf16_zero_B_gives_base_product():
    # B starts at 0, so the updated B equals the AdamW update itself, which at t = 1 is about
    # -lr * sign(g): the sign of near-zero gradient entries decides it.  The update is checked
    # on identical gradients in test_adamw_isolated_t3; here the layer outputs and moments.
    wl = W.custom("zero_B", 951, 384, 256, [8, 3], [100, 90], dtype="bf16", b_std=0.0)
    errs, got, want = _run(wl, keys=["Y", "dX", "H", "dH", "dAt", "dBt", "At", "mA", "vA", "mB", "vB"])
    # dA must vanish when B = 0 (Case 3 of the backward has B as a factor)
    assert all(np.max(np.abs(a)) == 0 for a in got["dAt"])


def test_repeat_calls_are_deterministic():
    wl = W.custom("repeat", 952, 256, 256, [8, 24], [150, 170], dtype="bf16")
    T = W.materialise(wl)
    r1 = G.GpuRun(wl, T, step=False)
    r2 = G.GpuRun(wl, T, step=False)
    try:
        for k in ("Y", "dX"):
            assert np.array_equal(r1.res[k], r2.res[k])
        for k in ("H", "dH", "dAt", "dBt"):
            assert all(np.array_equal(a, b) for a, b in zip(r1.res[k], r2.res[k]))
    finally:
        r1.close()
        r2.close()


def test_launch_overlap_does_not_change_results():
    """Programmatic dependent launch (the default for packs of this size) and strictly serial launches give bitwise
    identical outputs: every kernel waits for its predecessor before touching memory."""
    wl = W.custom("overlap", 954, 512, 384, [4, 64, 130], [300, 100, 150], dtype="bf16")
    T = W.materialise(wl)
    r1 = G.GpuRun(wl, T, step=True)
    r2 = G.GpuRun(wl, T, step=True, flags=M.MLORA_NO_OVERLAP)
    try:
        for k in ("Y", "dX"):
            assert np.array_equal(r1.res[k], r2.res[k])
        for k in ("H", "dH", "dAt", "dBt", "At", "Bt", "mA", "vA", "mB", "vB"):
            assert all(np.array_equal(a, b) for a, b in zip(r1.res[k], r2.res[k])), k
    finally:
        r1.close()
        r2.close()


def test_reuse_staging_gives_identical_results():
    """With MLORA_REUSE_STAGING the backward reuses the forward's shadows and images from the
    shared workspace; over two full steps (AdamW in between invalidates the reuse once) every
    output matches the plain path bitwise."""
    wl = W.custom("reuse", 956, 384, 512, [4, 64, 130], [300, 100, 150], dtype="bf16", b_std=0.05)
    T = W.materialise(wl)
    outs = []
    for flags in (0, M.MLORA_REUSE_STAGING):
        L = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At, Bt=T.Bt,
                         flags=flags)
        X, Wt, dY = G.to_dev(T.X, "bf16"), G.to_dev(T.Wt, "bf16"), G.to_dev(T.dY, "bf16")
        res = []
        for step in (1, 2):
            Y = L.forward(X, Wt)
            dX = L.backward(X, Wt, dY)
            L.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, step)
            torch.cuda.synchronize()
            res.append([G.from_dev(Y, "bf16"), G.from_dev(dX, "bf16")] + [a.cpu().numpy() for a in L.dAt + L.dBt + L.At])
        assert L.sync_status() == M.MLORA_OK
        outs.append(res)
        L.close()
    for a, b in zip(outs[0], outs[1]):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_adamw_isolated_t3():
    """The AdamW kernel alone on seeded gradients and moments (t = 3), so the update
    p' - p itself can be checked: at small t it is close to -lr * sign(g), which would
    amplify rounding differences in a gradient computed upstream."""
    wl = W.custom("adamw", 953, 264, 136, [3, 16, 40], [7, 9, 4], dtype="bf16")
    T = W.materialise(wl, with_dY=True)
    layer = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At, Bt=T.Bt)
    try:
        want = {}
        for i in range(wl.n_adapters):
            for which, p, g_t, m_t, v_t in (("A", layer.At[i], layer.dAt[i], layer.mA[i], layer.vA[i]),
                                            ("B", layer.Bt[i], layer.dBt[i], layer.mB[i], layer.vB[i])):
                shape = tuple(p.shape)
                g = W.optimizer_state(wl, which, i, shape, "g")
                m = W.optimizer_state(wl, which, i, shape, "m")
                v = W.optimizer_state(wl, which, i, shape, "v")
                g_t.copy_(torch.from_numpy(g))
                m_t.copy_(torch.from_numpy(m))
                v_t.copy_(torch.from_numpy(v))
                p0 = p.cpu().numpy().astype(np.float64)
                want[(which, i)] = (p0,) + orc.adamw(p0, g, m, v, 2e-3, 0.9, 0.95, 1e-8, 0.05, 3)
        layer.adamw(2e-3, 0.9, 0.95, 1e-8, 0.05, 3)
        torch.cuda.synchronize()
        for i in range(wl.n_adapters):
            for which, p, m_t, v_t in (("A", layer.At[i], layer.mA[i], layer.vA[i]),
                                       ("B", layer.Bt[i], layer.mB[i], layer.vB[i])):
                p0, pw, mw, vw = want[(which, i)]
                pg = p.cpu().numpy().astype(np.float64)
                assert G.rel_err(pg - p0, pw - p0) < 1e-4
                assert G.rel_err(pg, pw) < 1e-6
                assert G.rel_err(m_t.cpu().numpy(), mw) < 1e-6
                assert G.rel_err(v_t.cpu().numpy(), vw) < 1e-6
    finally:
        layer.close()


def test_device_wait_timeout_is_reported_and_context_survives():
    """A bounded device wait that runs out (test hook: a pipeline slot that no copy fills)
    surfaces as MLORA_ERR_TIMEOUT from mlora_sync_status, and the same process keeps working:
    a normal plan afterwards computes correct results."""
    wl = W.custom("timeout", 955, 256, 256, [8, 16], [200, 90], dtype="bf16")
    T = W.materialise(wl)
    bad = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At, Bt=T.Bt,
                       flags=M.MLORA_DEBUG_SHORT_TIMEOUT | M.MLORA_DEBUG_DROP_COPY)
    try:
        bad.forward(G.to_dev(T.X, "bf16"), G.to_dev(T.Wt, "bf16"))
        assert bad.sync_status() == M.MLORA_ERR_TIMEOUT
        assert bad.sync_status() == M.MLORA_OK          # the status word was read and cleared
    finally:
        bad.close()
    _run(wl)                                           # the context is still usable


@pytest.mark.parametrize("window", ["pairs", "single"])
def test_pair_kernel_wait_timeout_drains_and_context_survives(window):
    """The same for the forward's CTA-pair kernels (test hook: the first pair's even CTA arms its
    first slot for both CTAs' bytes but copies nothing).  With the shrink forced onto pairs both
    the shrink and the base GEMM give up; otherwise only the base GEMM does.  Each kernel's MMA
    wait runs out, its teardown waits (bounded) for the ring's outstanding copies, including the
    odd CTA's, before either CTA's shared memory goes away; the status reads MLORA_ERR_TIMEOUT once,
    and a normal plan afterwards computes correct results."""
    wl = W.custom("timeout_pairs", 956, 512, 384, [8, 64, 130], [300, 100, 150], dtype="bf16")
    T = W.materialise(wl)
    flags = M.MLORA_DEBUG_SHORT_TIMEOUT | M.MLORA_DEBUG_DROP_COPY_PAIRS
    flags |= M.MLORA_WINDOW_PAIRS if window == "pairs" else M.MLORA_WINDOW_SINGLE
    bad = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At, Bt=T.Bt,
                       flags=flags)
    try:
        bad.forward(G.to_dev(T.X, "bf16"), G.to_dev(T.Wt, "bf16"))
        assert bad.sync_status() == M.MLORA_ERR_TIMEOUT
        assert bad.sync_status() == M.MLORA_OK
    finally:
        bad.close()
    _run(wl)


@pytest.mark.parametrize("grouped", [False, True], ids=["one_group", "qkv_groups"])
def test_adamw_shadow_refresh_matches_repacking(grouped):
    """Three steps with MLORA_REUSE_STAGING and mlora_adamw_ws (the forward reuses the shadows the
    AdamW step refreshed) give bit-identical results to three steps that repack every time."""
    if grouped:
        wl = W.custom_grouped("shadow_refresh_g", 931, 512, [256, 64, 64], [[8, 8, 8], [64, 16, 1], [3, 128, 32]],
                              [200, 56, 300], b_std=0.05)
    else:
        wl = W.custom("shadow_refresh", 930, 512, 640, [1, 7, 64, 256], [200, 56, 300, 17], b_std=0.05)
    T = W.materialise(wl)
    X, dY = G.to_dev(T.X, "bf16"), G.to_dev(T.dY, "bf16")
    Wt = G.to_dev(T.Wt, "bf16")
    outs = []
    for flags, refresh in ((M.MLORA_REUSE_STAGING, True), (0, False)):
        layer = G.make_layer(wl, T, flags)
        try:
            res = []
            for step in range(1, 4):
                Y = layer.forward(X, Wt)
                dX = layer.backward(X, Wt, dY)
                layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, step, refresh_shadows=refresh)
                res.append((Y.clone(), dX.clone()))
            torch.cuda.synchronize()
            assert layer.sync_status() == M.MLORA_OK
            outs.append((res, [a.clone() for a in layer.At], [b.clone() for b in layer.Bt]))
        finally:
            layer.close()
    (r1, A1, B1), (r2, A2, B2) = outs
    for (y1, x1), (y2, x2) in zip(r1, r2):
        assert torch.equal(y1, y2) and torch.equal(x1, x2)
    assert all(torch.equal(a, b) for a, b in zip(A1, A2))
    assert all(torch.equal(a, b) for a, b in zip(B1, B2))


def test_cuda_graph_replay_matches_eager_steps():
    """One step (forward, backward, AdamW refreshing the shadows) captured in a CUDA graph after a
    warm-up step and replayed twice gives bit-identical results to running the same steps eagerly
    (launches with programmatic dependent launch are captured as such)."""
    wl = W.custom("graph_replay", 933, 512, 640, [1, 7, 64, 256], [200, 56, 300, 17], b_std=0.05)
    T = W.materialise(wl)
    X, dY = G.to_dev(T.X, "bf16"), G.to_dev(T.dY, "bf16")
    Wt = G.to_dev(T.Wt, "bf16")
    results = []
    for use_graph in (False, True):
        layer = G.make_layer(wl, T, M.MLORA_REUSE_STAGING)
        Y = torch.empty((wl.N, wl.d_out), dtype=torch.bfloat16, device="cuda")
        dX = torch.empty((wl.N, wl.d_in), dtype=torch.bfloat16, device="cuda")
        step = [0]

        def one_step():
            step[0] += 1
            layer.forward(X, Wt, Y)
            layer.backward(X, Wt, dY, dX)
            layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, 1)   # fixed t: replays are identical

        try:
            one_step()                                   # warm-up: packs and leaves the shadows current
            torch.cuda.synchronize()
            if use_graph:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    one_step()
                torch.cuda.current_stream().wait_stream(s)
                graph.replay()
                graph.replay()
            else:
                one_step()
                one_step()
            torch.cuda.synchronize()
            assert layer.sync_status() == M.MLORA_OK
            results.append((Y.clone(), dX.clone(), [a.clone() for a in layer.At], [b.clone() for b in layer.Bt]))
        finally:
            layer.close()
    # capturing records without running: both sides applied the step three times (warm-up + 2)
    (y1, x1, a1, b1), (y2, x2, a2, b2) = results
    assert torch.equal(y1, y2) and torch.equal(x1, x2)
    assert all(torch.equal(p, q) for p, q in zip(a1, a2)) and all(torch.equal(p, q) for p, q in zip(b1, b2))


def test_autograd_module_matches_direct_calls():
    """PackedLoRALinear through torch.autograd gives the same Y, dX (as X.grad), adapter gradients
    and AdamW step as calling the layer directly."""
    from adapter_gemm_packed_gb300.layer import PackedLoRALinear
    wl = W.custom("autograd", 934, 512, 640, [1, 7, 64, 256], [200, 56, 300, 17], b_std=0.05)
    T = W.materialise(wl)
    Wt = G.to_dev(T.Wt, "bf16")
    dY = G.to_dev(T.dY, "bf16")
    direct = G.make_layer(wl, T, M.MLORA_REUSE_STAGING)
    viaag = G.make_layer(wl, T, M.MLORA_REUSE_STAGING)
    try:
        X = G.to_dev(T.X, "bf16")
        Y1 = direct.forward(X, Wt)
        dX1 = direct.backward(X, Wt, dY)
        direct.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, 1)
        mod = PackedLoRALinear(viaag, Wt)
        Xg = G.to_dev(T.X, "bf16").requires_grad_(True)
        Y2 = mod(Xg)
        Y2.backward(dY)
        mod.step(wl.lr, (wl.beta1, wl.beta2), wl.eps, wl.weight_decay)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2.detach()) and torch.equal(dX1, Xg.grad)
        for k in ("dAt", "dBt", "At", "Bt"):
            assert all(torch.equal(a, b) for a, b in zip(getattr(direct, k), getattr(viaag, k))), k
    finally:
        direct.close()
        viaag.close()


def test_two_plans_on_two_threads_and_streams():
    """Two plans driven at once from two host threads on their own streams (the library's host
    code runs concurrently: ctypes releases the GIL) match the same plans run one after the other."""
    import threading
    cases = [W.custom("thr_a", 935, 512, 640, [1, 7, 64, 256], [200, 56, 300, 17], b_std=0.05),
             W.custom("thr_b", 936, 384, 256, [16, 128, 8], [256, 384, 130], b_std=0.05)]
    data = []
    for wl in cases:
        T = W.materialise(wl)
        data.append((wl, T, G.to_dev(T.X, "bf16"), G.to_dev(T.dY, "bf16"), G.to_dev(T.Wt, "bf16")))

    def run(i, stream, out):
        wl, T, X, dY, Wt = data[i]
        layer = G.make_layer(wl, T, M.MLORA_REUSE_STAGING)
        try:
            with torch.cuda.stream(stream):
                for step in range(1, 4):
                    Y = layer.forward(X, Wt, stream=stream)
                    dX = layer.backward(X, Wt, dY, stream=stream)
                    layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, step, stream=stream)
            stream.synchronize()
            assert layer.sync_status(stream) == M.MLORA_OK
            out[i] = (Y.clone(), dX.clone(), [a.clone() for a in layer.At])
        finally:
            layer.close()

    seq = [None, None]
    for i in range(2):
        run(i, torch.cuda.Stream(), seq)
    par = [None, None]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    threads = [threading.Thread(target=run, args=(i, streams[i], par)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for a, b in zip(seq, par):
        assert b is not None
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert all(torch.equal(x, y) for x, y in zip(a[2], b[2]))


def _random_wl(seed):
    g = np.random.default_rng(5000 + seed)
    n_jobs = int(g.integers(1, 9))
    ns = [int(n) for n in g.choice([1, 7, 64, 127, 128, 129, 200, 300], size=n_jobs)]
    d_in = 64 * int(g.integers(1, 9))
    if seed % 3 == 2:   # a shared-input pack of two or three projections
        widths = [8 * int(w) for w in g.integers(2, 40, size=int(g.integers(2, 4)))]
        ranks_jg = [[int(r) for r in g.choice([1, 4, 8, 16, 32, 64, 128], size=len(widths))] for _ in ns]
        return W.custom_grouped(f"rand_g{seed}", 940 + seed, d_in, widths, ranks_jg, ns, b_std=0.05)
    d_out = 8 * int(g.integers(2, 80))
    ranks = [int(r) for r in g.choice([1, 3, 8, 16, 33, 64, 128, 256], size=n_jobs)]
    return W.custom(f"rand_{seed}", 940 + seed, d_in, d_out, ranks, ns, b_std=0.05, w_std=0.05)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_vs_oracle(seed):
    """Seeded random job tables (1-8 jobs of 1-300 tokens, ranks 1-256, ragged widths, every third a
    shared-input pack), the shrink / dH engine alternating between pairs and single CTAs."""
    wl = _random_wl(seed)
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, flags=M.MLORA_WINDOW_PAIRS if seed % 2 else M.MLORA_WINDOW_SINGLE)
    try:
        assert run.status_after_backward == M.MLORA_OK
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16"])
    finally:
        run.close()


@pytest.mark.parametrize("grouped", [False, True], ids=["one_group", "qkv_groups"])
def test_wgrad_items_cut_across_ctas_vs_oracle(grouped):
    """dA / dB items whose tokens the schedule cuts across CTAs (each part parks fp32 sums, the
    last part to arrive adds them in part order): long jobs next to short ones, so that items run
    as 3 or more parts, in a plain pack and in a shared-input pack; every output against the oracle,
    twice in a row bitwise (the partial sums' order does not depend on arrival order)."""
    ns = [6000, 300, 4100, 64]
    if grouped:
        wl = W.custom_grouped("wgrad_cut_g", 962, 1024, [512, 128, 128], [[16, 8, 8], [64, 16, 16], [128, 32, 8],
                                                                          [8, 8, 1]], ns, b_std=0.05)
    else:
        wl = W.custom("wgrad_cut", 961, 1024, 768, [16, 64, 128, 8], ns, b_std=0.05, w_std=0.05)
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, step=False)
    try:
        assert run.status_after_backward == M.MLORA_OK
        for what in (M.MLORA_Q_WGRAD_A, M.MLORA_Q_WGRAD_B):
            items = np.array(run.layer.describe(what)).reshape(-1, 9)
            assert items[:, 7].max() >= 3
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16"], ["dAt", "dBt", "dX", "Y", "H", "dH"])
        first = [a.clone() for a in run.layer.dAt] + [b.clone() for b in run.layer.dBt]
        run.layer.backward(run.X, run.Wt, run.dY)
        torch.cuda.synchronize()
        assert run.layer.sync_status() == M.MLORA_OK
        again = list(run.layer.dAt) + list(run.layer.dBt)
        assert all(torch.equal(a, b) for a, b in zip(first, again))
    finally:
        run.close()


PAIR_CUT_CASES = {
    # three one-job pair tiles of two chunks, 64 K slices each way: every item in four pieces
    "even": lambda: W.custom("pair_cut", 963, 4096, 4096, [128, 128, 128], [256, 256, 256], b_std=0.05, w_std=0.05),
    # several jobs per pair tile (items of four chunks and a padded pair), ragged ranks and
    # tokens, dH 32 slices against the shrink's 64
    "ragged": lambda: W.custom("pair_cut_r", 964, 4096, 2048, [3, 64, 200, 17, 128], [100, 300, 57, 250, 40],
                               b_std=0.05, w_std=0.05),
    # a shared-input pack: the first job's window is six chunks, so its second item holds only the
    # k / v adapters' columns and its dH reads (and is cut within) their d_out slices 32..63
    "qkv_groups": lambda: W.custom_grouped("pair_cut_g", 965, 4096, [2048, 1024, 1024],
                                           [[256, 64, 64], [32, 16, 16], [16, 8, 8]], [256, 200, 250],
                                           b_std=0.05),
}


@pytest.mark.parametrize("name", sorted(PAIR_CUT_CASES))
def test_pair_items_cut_along_k_vs_oracle(name):
    """CTA-pair shrink / dH items that the per-pair schedule cuts along K (few items for the pairs:
    every item in several pieces, each parking fp32 sums; the last piece to arrive adds them in
    piece order and writes H / dH and the images): every output against the oracle, and a second
    forward + backward bitwise equal to the first."""
    wl = PAIR_CUT_CASES[name]()
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, step=False, flags=M.MLORA_WINDOW_PAIRS)
    try:
        assert run.status_after_backward == M.MLORA_OK
        # entries: product (0 shrink, 1 dH), pair, tile pair, first chunk, chunks, first K slice,
        # K slices, piece, pieces
        items = np.array(run.layer.describe(M.MLORA_Q_WINDOW_PAIRS))[1:].reshape(-1, 9)
        assert items[:, 8].min() >= 2          # every item cut, in both products
        if name == "qkv_groups":
            assert ((items[:, 0] == 1) & (items[:, 5] >= 32)).any()   # a dH piece inside the k / v slices
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16"], ["Y", "dX", "H", "dH", "dAt", "dBt"])
        first = [t.clone() for t in (run.layer.H, run.layer.dH)]
        run.layer.forward(run.X, run.Wt)
        run.layer.backward(run.X, run.Wt, run.dY)
        torch.cuda.synchronize()
        assert run.layer.sync_status() == M.MLORA_OK
        assert all(torch.equal(a, b) for a, b in zip(first, (run.layer.H, run.layer.dH)))
    finally:
        run.close()


@pytest.mark.parametrize("reuse", [False, True], ids=["repack", "reuse_staging"])
def test_three_training_steps_vs_oracle(reuse):
    """Three steps of forward, backward and AdamW (t = 1, 2, 3) with fresh X and dY each step: the
    masters, moments and (with MLORA_REUSE_STAGING) the bf16 shadows refreshed by the AdamW step carry
    over between steps as the oracle's state does.  Checked after the third step: Y, dX, H, dH, dA,
    dB of that step and every adapter's A, B, m, v."""
    wl = W.custom("three_steps", 906, 512, 384, [8, 64, 3, 24], [200, 77, 300, 129], w_std=0.05, b_std=0.05)
    T = W.materialise(wl)
    layer = G.make_layer(wl, T, flags=M.MLORA_REUSE_STAGING if reuse else 0)
    Wt = G.to_dev(T.Wt, wl.dtype)
    Wm = W.rows_as_f64(T.Wt, wl.dtype).T
    J = len(wl.ranks)
    A = [T.At[j].astype(np.float64).T for j in range(J)]          # d_in x r
    B = [T.Bt[j].astype(np.float64).T for j in range(J)]          # r x d_out
    mA = [np.zeros_like(a) for a in A]
    vA = [np.zeros_like(a) for a in A]
    mB = [np.zeros_like(b) for b in B]
    vB = [np.zeros_like(b) for b in B]
    for t in (1, 2, 3):
        Xb = W.to_bf16_bits(W.normal_f32(906, 100 + 2 * t, wl.N * wl.d_in, 1.0).reshape(wl.N, wl.d_in))
        dYb = W.to_bf16_bits(W.normal_f32(906, 101 + 2 * t, wl.N * wl.d_out, 1.0).reshape(wl.N, wl.d_out))
        X, dY = G.to_dev(Xb, wl.dtype), G.to_dev(dYb, wl.dtype)
        Y = layer.forward(X, Wt)
        dX = layer.backward(X, Wt, dY)
        torch.cuda.synchronize()
        got = dict(Y=G.from_dev(Y, wl.dtype), dX=G.from_dev(dX, wl.dtype),
                   H=[h.cpu().numpy().astype(np.float64) for h in layer.h_blocks()],
                   dH=[h.cpu().numpy().astype(np.float64) for h in layer.h_blocks(layer.dH)],
                   dAt=[a.cpu().numpy().astype(np.float64) for a in layer.dAt],
                   dBt=[b.cpu().numpy().astype(np.float64) for b in layer.dBt])
        layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, t)
        segs = [orc.Seg(o, n, A[j], B[j], wl.alphas[j]) for j, (o, n) in enumerate(zip(wl.offsets, wl.n_tokens))]
        Xf, dYf = W.rows_as_f64(Xb, wl.dtype), W.rows_as_f64(dYb, wl.dtype)
        Yo, Ho = orc.forward(Xf, Wm, segs)
        dXo, dAo, dBo, dHo = orc.backward(Xf, Wm, dYf, segs)
        for j in range(J):
            A[j], mA[j], vA[j] = orc.adamw(A[j], dAo[j], mA[j], vA[j], wl.lr, wl.beta1, wl.beta2, wl.eps,
                                           wl.weight_decay, t)
            B[j], mB[j], vB[j] = orc.adamw(B[j], dBo[j], mB[j], vB[j], wl.lr, wl.beta1, wl.beta2, wl.eps,
                                           wl.weight_decay, t)
    torch.cuda.synchronize()
    assert layer.sync_status() == M.MLORA_OK
    got.update(At=[a.cpu().numpy().astype(np.float64) for a in layer.At],
               Bt=[b.cpu().numpy().astype(np.float64) for b in layer.Bt],
               mA=[a.cpu().numpy().astype(np.float64) for a in layer.mA],
               vA=[a.cpu().numpy().astype(np.float64) for a in layer.vA],
               mB=[b.cpu().numpy().astype(np.float64) for b in layer.mB],
               vB=[b.cpu().numpy().astype(np.float64) for b in layer.vB])
    want = dict(Y=Yo, dX=dXo, H=Ho, dH=dHo, dAt=[a.T for a in dAo], dBt=[b.T for b in dBo],
                At=[a.T for a in A], Bt=[b.T for b in B], mA=[m.T for m in mA], vA=[v.T for v in vA],
                mB=[m.T for m in mB], vB=[v.T for v in vB])
    G.compare(got, want, G.TOL[wl.dtype])
    layer.close()
