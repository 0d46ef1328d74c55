"""GPU parity of the gate GEMM and the fused router epilogue against the
oracle, through the C ABI, on every workload: the tiny router, decode
(T = 1, 8, 64), prefill (T = 4096), the adversarial large batch (T = 16384,
E = 384) and the wide-N raw head (N = 129280, k = 1 and 8), plus ragged
shapes, both kernels (single-launch decode and tensor-core), exact integer
logits, determinism, CUDA-graph replay and workspace reuse."""

import os
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from oracle import formats, quantize as Q, gemm, router, compare  # noqa: E402
from gpu_util import Case, to_device, as_f32  # noqa: E402

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))

TC = 2       # NVR_FLAG_FORCE_TENSOR_CORE
DEC = 4      # NVR_FLAG_FORCE_DECODE
K2, K4, K8 = 8, 16, 32   # NVR_FLAG_SPLIT_K_2/4/8: K split over that many CTAs
SPN = 64     # NVR_FLAG_SPLIT_N: the N-split tensor-core kernel


def _logits(case, flags):
    import nvfp4_router_gate_gb300 as R
    out = R.router_gate_logits(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, flags=flags)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,T,flags", [("tiny", 4, DEC), ("tiny", 4, TC), ("decode", 8, DEC),
                                          ("decode", 8, TC), ("prefill", 300, TC),
                                          ("prefill", 300, K2), ("prefill", 300, K4),
                                          ("prefill", 300, K8), ("prefill", 300, SPN),
                                          ("adversarial", 40, TC)])
def test_logits_within_tolerance(name, T, flags):
    case = Case(WL.WORKLOADS[name].with_T(T))
    g = _logits(case, flags)
    L, B = case.oracle_rows(np.arange(T))
    assert compare.check_logits(g, L, B) == 0
    # much tighter than the contract in practice: report the worst relative error
    rel = np.abs(g - L) / (compare.LOGIT_ABS_FRAC * B + np.abs(L) + 1e-30)
    assert rel.max() < 1e-4


def test_prefill_logits_full_size_default_plan():
    """All 4096 x 256 logits of the prefill batch on the plan a default call
    takes (one launch; at T = 4096 on a GB300: 112-row tiles, K split over 4
    CTAs, no clusters), element by element under the logit tolerance."""
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["prefill"]
    case = Case(w)
    R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, w.k, w.routed_scaling)
    plan_topk = R.last_router_plan()
    g = _logits(case, 0)
    assert R.last_router_plan() == plan_topk and plan_topk["sequence"] == "fused", plan_topk
    L, B = case.oracle_rows(np.arange(w.T))
    assert compare.check_logits(g, L, B) == 0
    rel = np.abs(g - L) / (compare.LOGIT_ABS_FRAC * B + np.abs(L) + 1e-30)
    assert rel.max() < 1e-4


def _grid_operands(rng, rows, D, amax_block):
    """Inputs whose NVFP4 quantization is exact: gsa = 1 (one element 2688 =
    6 * 448 alone in block `amax_block` of row 0) and block scales 2**b,
    b in [-1, 1], with a +-6 leading every other block."""
    vals = formats.decode_e2m1(rng.integers(0, 16, (rows, D)))
    vals[:, ::16] = 6.0 * rng.choice([-1, 1], (rows, D // 16))
    b = rng.integers(-1, 2, (rows, D // 16))
    x = vals * np.repeat(2.0 ** b, 16, axis=1)
    x[0, 16 * amax_block:16 * (amax_block + 1)] = 0.0
    x[0, 16 * amax_block] = 2688.0
    return x.astype(np.float32)


@pytest.mark.parametrize("flags", [DEC, TC, K2, K4, K8, SPN])
def test_exact_integer_logits(flags):
    """Grid-valued operands: products are multiples of 1/16 and every partial
    sum stays below 2**20 in magnitude, so any fp32 summation order is exact
    and the GPU logits must equal the oracle's bits."""
    import nvfp4_router_gate_gb300 as R
    rng = np.random.default_rng(21)
    T, N, D = 8, 136, 512
    x = _grid_operands(rng, T, D, 0)
    W = _grid_operands(rng, N, D, 1)      # the two 2688s never meet in one product
    xd, Wd = to_device(x, "f32"), to_device(W, "f32")
    wf, ws, wg = R.nvfp4_pack_weight(Wd)
    out = R.router_gate_logits(xd, wf, ws, wg, flags=flags)
    torch.cuda.synchronize()
    xq, xs, xg = Q.quantize(x)
    wq, wsb, wgg = Q.quantize(W)
    assert xg == 1.0 and wgg == 1.0
    L, _ = gemm.logits(xq, xs, xg, wq, wsb, wgg)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), L)


@pytest.mark.parametrize("flags", [DEC, TC])
def test_tiny_router(flags):
    case = Case(WL.WORKLOADS["tiny"])
    ids, w = case.run(flags)
    res = case.check(ids, w, np.arange(case.w.T))
    assert compare.topk_ok(res) and res["exempt_rows"] == 0, res


@pytest.mark.parametrize("T", [1, 8, 64])
def test_decode_router(T):
    case = Case(WL.WORKLOADS["decode"].with_T(T))
    ids, w = case.run()
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res
    if T <= 8:
        ids2, w2 = case.run(TC)                      # the other kernel agrees too
        res2 = case.check(ids2, w2, np.arange(T))
        assert compare.topk_ok(res2), res2


def test_prefill_router_odd_tile_count():
    """T = 5000: 40 token tiles, so the planner's K-split is not a power of two
    and the fused kernel rounds it down (sampled rows, including the ragged
    last tile)."""
    case = Case(WL.WORKLOADS["prefill"].with_T(5000))
    ids, w = case.run()
    rows = np.unique(np.concatenate([np.arange(0, 5000, 97), np.arange(4990, 5000), [127, 128, 4991]]))
    res = case.check(ids, w, rows)
    assert compare.topk_ok(res), res


def test_prefill_router_all_rows():
    """Every row of the T = 4096 prefill batch on the default one-launch plan,
    and the global scale that launch computed itself (bit-exact)."""
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["prefill"]
    case = Case(w)
    ws = R.new_workspace(R.router_gate_workspace_size(w.T, w.D, w.N, w.k))
    ids, wts = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, w.k,
                                  w.routed_scaling, w.raw, workspace=ws)
    torch.cuda.synchronize()
    assert R.last_router_plan()["sequence"] == "fused"
    gsa = R.router_gate_x_gsa(ws).item()
    assert np.float32(gsa).view(np.uint32) == Q.global_scale(case.x32).view(np.uint32)
    res = case.check(ids.cpu().numpy(), wts.cpu().numpy(), np.arange(w.T))
    assert compare.topk_ok(res), res


@pytest.mark.parametrize("T", [129, 300])
def test_ragged_batches_all_rows(T):
    case = Case(WL.WORKLOADS["prefill"].with_T(T))
    ids, w = case.run()
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res


def test_adversarial_router():
    """Every row of the T = 16384, E = 384 adversarial batch."""
    case = Case(WL.WORKLOADS["adversarial"])
    ids, w = case.run()
    res = case.check(ids, w, np.arange(case.w.T))
    assert compare.topk_ok(res), res
    # all-zero rows (t % 4 == 1): every logit is exactly 0, so the ids are 0..7
    # and each weight is routed_scaling / 8
    zero = np.arange(1, 16384, 4)
    assert np.all(ids[zero] == np.arange(8))
    assert np.allclose(w[zero], 2.5 / 8, atol=1e-6)
    # 1e4 rows saturate the sigmoid: weights are 2.5/8 up to 1e-5
    big = np.arange(2, 16384, 4)
    assert np.all(np.abs(w[big].sum(axis=1) - 2.5) < 1e-4)


def test_adversarial_tie_probe():
    """Experts 2j+1 duplicate 2j: exact ties in every row must keep the lower id first."""
    case = Case(WL.Workload("tie_probe", 256, 7168, 384, 8, 2.5, False, "bf16", "adversarial", 0.02,
                            "zero", tie_probe=True))
    ids, w = case.run()
    res = case.check(ids, w, np.arange(256))
    assert compare.topk_ok(res), res
    for row in ids:
        pos = {int(e): i for i, e in enumerate(row)}
        for e, i in pos.items():
            if e < 16 and e % 2 == 1 and (e - 1) in pos:
                assert pos[e - 1] < i                # the even copy comes first


GOLDEN_WIDE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "wide_n_expected.npz")


@pytest.mark.parametrize("k", [1, 8])
def test_wide_n_raw_head(k):
    """All 32 tokens of the N = 129280 raw head against the oracle's stored
    answer (tests/golden/make_wide_n_expected.py: quantizing the weight on the
    CPU takes minutes)."""
    if not os.path.exists(GOLDEN_WIDE):
        pytest.skip("tests/golden/wide_n_expected.npz not generated")
    gold = np.load(GOLDEN_WIDE)
    w = WL.WORKLOADS["wide_n"].with_k(k)
    case = Case(w, with_oracle_w=False)
    import make_wide_n_expected as gen
    if gen.input_digest(w) != str(gold["digest"]):
        pytest.fail("the seeded generator no longer reproduces the stored inputs")
    assert case.w_gsa.item() == float(gold["w_gsa"])
    ids, wts = case.run()
    res = compare.check_topk_candidates(ids, wts, gold["ids"], gold["logits"], gold["bounds"],
                                        gold["rest_max"], raw=True)
    assert compare.topk_ok(res), res


def test_determinism_and_graph_replay():
    import nvfp4_router_gate_gb300 as R
    for T in (1, 300):
        w = WL.WORKLOADS["decode"].with_T(T) if T == 1 else WL.WORKLOADS["prefill"].with_T(T)
        gate = R.RouterGate(to_device(WL.make_w(w), w.dtype), torch.from_numpy(WL.make_bias(w)).cuda(),
                            k=8, routed_scaling=2.5, max_tokens=T)
        x = to_device(WL.make_x(w), w.dtype)
        ids0, w0 = [t.clone() for t in gate(x)]
        ids1, w1 = [t.clone() for t in gate(x)]
        assert torch.equal(ids0, ids1) and torch.equal(w0, w1)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            gate(x)                                  # warm up on the capture stream
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            gate(x)
        gate.ids.zero_()
        for _ in range(20):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(gate.ids[:T], ids0) and torch.equal(gate.weights[:T], w0)
        assert R.nvr_read_device_status(gate.workspace) == 0


def test_steady_state_calls_neither_sync_nor_allocate():
    """A resident router's calls make no synchronising torch call (the sync
    debug mode raises on one) and allocate nothing (the caching allocator's
    count stays put over many calls): nothing hidden between the host and a
    CUDA graph, decode and prefill alike."""
    import nvfp4_router_gate_gb300 as R
    for T in (1, 300):
        w = WL.WORKLOADS["decode"].with_T(T) if T == 1 else WL.WORKLOADS["prefill"].with_T(T)
        gate = R.RouterGate(to_device(WL.make_w(w), w.dtype), torch.from_numpy(WL.make_bias(w)).cuda(),
                            k=8, routed_scaling=2.5, max_tokens=T)
        x = to_device(WL.make_x(w), w.dtype)
        gate(x)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        torch.cuda.set_sync_debug_mode("error")
        try:
            for _ in range(200):
                gate(x)
        finally:
            torch.cuda.set_sync_debug_mode("default")
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        assert R.nvr_read_device_status(gate.workspace) == 0


def test_workspace_reuse_across_shapes():
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["prefill"]
    case = Case(w.with_T(600))
    ws = R.new_workspace(R.router_gate_workspace_size(600, 7168, 256, 8))
    for T in (600, 1, 9, 128, 600, 16):
        x = case.x_dev[:T].contiguous()
        ids, wt = R.router_gate_topk(x, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                                     workspace=ws)
        torch.cuda.synchronize()
        sub = Case.__new__(Case)
        sub.__dict__.update(case.__dict__)
        sub.x32 = case.x32[:T]
        sub.w = w.with_T(T)
        res = sub.check(ids.cpu().numpy(), wt.cpu().numpy(), np.arange(T))
        assert compare.topk_ok(res), (T, res)
    assert R.nvr_read_device_status(ws) == 0


def test_gpu_argument_errors():
    import nvfp4_router_gate_gb300 as R
    case = Case(WL.WORKLOADS["tiny"])
    with pytest.raises(R.RouterError):
        R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, None, k=17)
    # the wide head needs the tensor-core path: forcing the decode kernel is refused
    big = torch.zeros((32, 7168), dtype=torch.bfloat16, device="cuda")
    wf = torch.zeros((20000, 3584), dtype=torch.uint8, device="cuda")
    wsf = torch.zeros(R.nvr_sf_bytes(20000, 7168, "tiled"), dtype=torch.uint8, device="cuda")
    with pytest.raises(R.RouterError, match="unsupported"):
        R.router_gate_topk(big, wf, wsf, case.w_gsa, None, k=1, flags=DEC)


@pytest.mark.parametrize("kflag", [TC, SPN])
def test_bounded_wait_timeout_reports_status(kflag):
    """Failure detection without a GPU fault: with the test stall hook the
    tensor-core kernel's MMA issuer issues nothing, its pipeline waits run out
    after about a second, the kernel records NVR_ERR_TIMEOUT in the workspace
    status word and returns.  The context stays usable: after re-zeroing the
    workspace the next call routes correctly."""
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    case = Case(WL.WORKLOADS["decode"].with_T(8))
    ws = R.new_workspace(R.router_gate_workspace_size(8, 7168, 256, 8))
    R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                       workspace=ws, flags=kflag | _native.NVR_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == _native.NVR_ERR_TIMEOUT
    ws.zero_()
    ids, w = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                                workspace=ws, flags=kflag)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == 0
    res = case.check(ids.cpu().numpy(), w.cpu().numpy(), np.arange(8))
    assert compare.topk_ok(res), res


# ---------------------------------------------------------------- kernel choices
# Heads of up to 256 experts run on the K-split GEMM (S CTAs per 128-token
# tile, fp32 partial logits summed by the epilogue kernel); S = 2, 4, 8 and
# the N-split kernel are forced here on the same inputs.

@pytest.mark.parametrize("flags", [K2, K4, K8, SPN])
@pytest.mark.parametrize("T", [129, 300])
def test_kernel_choices_all_rows(T, flags):
    case = Case(WL.WORKLOADS["prefill"].with_T(T))
    ids, w = case.run(flags)
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res


@pytest.mark.parametrize("flags", [K2, K4, K8])
@pytest.mark.parametrize("k", [1, 3, 16])
def test_split_k_k_values(flags, k):
    """k = 1 (a plain arg-max), k = 3 and the largest k = 16."""
    case = Case(WL.WORKLOADS["decode"].with_T(64).with_k(k))
    ids, w = case.run(flags)
    res = case.check(ids, w, np.arange(64))
    assert compare.topk_ok(res), res


@pytest.mark.parametrize("flags", [TC, K2, K4, K8])
def test_split_k_ties_and_saturated_rows(flags):
    """The adversarial rows on a 256-expert head: all-zero rows tie all 256
    keys at 0.5 and saturated rows tie many at 1.0; lower ids must win every
    tie."""
    w = WL.Workload("adversarial_256", 512, 7168, 256, 8, 2.5, False, "bf16", "adversarial", 0.02, "zero")
    case = Case(w)
    ids, wt = case.run(flags)
    res = case.check(ids, wt, np.arange(512))
    assert compare.topk_ok(res), res
    zero = np.arange(1, 512, 4)
    assert np.all(ids[zero] == np.arange(8))
    assert np.allclose(wt[zero], 2.5 / 8, atol=1e-6)


@pytest.mark.parametrize("flags", [TC, K2, K8])
def test_split_k_tie_probe(flags):
    w = WL.Workload("tie_probe_256", 256, 7168, 256, 8, 2.5, False, "bf16", "adversarial", 0.02,
                    "zero", tie_probe=True)
    case = Case(w)
    ids, wt = case.run(flags)
    res = case.check(ids, wt, np.arange(256))
    assert compare.topk_ok(res), res
    for row in ids:
        pos = {int(e): i for i, e in enumerate(row)}
        for e, i in pos.items():
            if e < 16 and e % 2 == 1 and (e - 1) in pos:
                assert pos[e - 1] < i


@pytest.mark.parametrize("flags", [K2, K4, K8])
def test_split_k_raw_head(flags):
    """RAW mode on a 200-expert head (the second 128-expert half is partial)."""
    w = WL.Workload("raw_200", 64, 7168, 200, 8, 1.0, True, "bf16", "normal", 0.02, "none")
    case = Case(w)
    ids, wt = case.run(flags)
    res = case.check(ids, wt, np.arange(64))
    assert compare.topk_ok(res), res


def test_split_k_flag_rejects_wide_heads():
    import nvfp4_router_gate_gb300 as R
    big = torch.zeros((32, 512), dtype=torch.bfloat16, device="cuda")
    wf = torch.zeros((300, 256), dtype=torch.uint8, device="cuda")
    wsf = torch.zeros(R.nvr_sf_bytes(300, 512, "tiled"), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(R.RouterError, match="unsupported"):
        R.router_gate_topk(big, wf, wsf, g, None, k=8, flags=K4)


# One launch or two: when every token tile's cluster fits on the GPU at once,
# the fused kernel computes max|x| itself (a grid barrier in the workspace);
# otherwise the amax kernel runs first.  With S = 8 forced, 20 tiles need 20
# clusters of 8 CTAs, more than a 152-SM GB300 holds (19): the two-launch path.

@pytest.mark.parametrize("flags", [0, K8])
def test_prefill_one_launch_and_two_launch_paths(flags):
    case = Case(WL.WORKLOADS["prefill"].with_T(2560))
    ids, w = case.run(flags)
    rows = np.concatenate([np.arange(0, 2560, 23), [2559]])
    res = case.check(ids, w, rows)
    assert compare.topk_ok(res), res


def test_prefill_one_launch_back_to_back_calls_on_one_workspace():
    """Five calls queued back to back on one workspace, on inputs whose
    magnitudes differ by up to 2^14: each call must quantize with its own
    max|x| (the barrier's maximum slot alternates between calls and the next
    call's slot is reset by the last CTA to arrive)."""
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["prefill"].with_T(1024)
    case = Case(w)
    ws = R.new_workspace(R.router_gate_workspace_size(w.T, w.D, w.N, w.k))
    rows = np.arange(0, w.T, 37)
    outs = []
    for scale in (1.0, 64.0, 2.0 ** -8, 3.0, 1.0):
        bits = WL.float32_to_bf16_bits((case.x32 * np.float32(scale)).astype(np.float32))
        ids, wts = R.router_gate_topk(to_device(bits, "bf16"), case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev,
                                      w.k, w.routed_scaling, w.raw, workspace=ws)
        outs.append((scale, bits, ids, wts))
    torch.cuda.synchronize()
    for scale, bits, ids, wts in outs:
        x32 = WL.bf16_bits_to_float32(bits)
        gsa = Q.global_scale(x32)
        xq, xs, _ = Q.quantize(x32[rows], gsa=gsa)
        L, B = gemm.logits(xq, xs, gsa, case.wq, case.ws, case.wg)
        keys = router.selection_keys(L, case.bias, w.raw)
        res = compare.check_topk(ids.cpu().numpy()[rows], wts.cpu().numpy()[rows], L, B, keys, case.bias,
                                 w.routed_scaling, w.raw)
        assert compare.topk_ok(res), (scale, res)


def test_prefill_plans_with_and_without_clusters():
    """Batch sizes whose plans differ: K-split tiles whose CTAs form a cluster
    (small grids) and, where the device holds more CTAs without clusters than
    in whole clusters, tiles whose CTAs meet at a workspace barrier (112-row
    tiles at T = 4096).  Every plan must route like the oracle, ragged last
    tile included."""
    import nvfp4_router_gate_gb300 as R
    seen = set()
    for T in (64, 256, 1000, 1024, 2048, 3001, 4096):
        case = Case(WL.WORKLOADS["prefill"].with_T(T))
        ids, w = case.run(0)
        plan = R.last_router_plan()
        assert plan["sequence"] in ("fused", "amax+fused"), (T, plan)
        seen.add((plan["sequence"], plan["clustered"]))
        rows = np.concatenate([np.arange(0, T, 41), np.arange(max(T - 20, 0), T)])
        res = case.check(ids, w, np.unique(rows))
        assert compare.topk_ok(res), (T, plan, res)
    assert ("fused", True) in seen and ("fused", False) in seen, seen


def test_prefill_mixed_plans_back_to_back_on_one_workspace():
    """Calls of different sizes -- with and without clusters, 128- and
    112-row tiles -- queued back to back on one workspace sized for the
    largest: the tile barriers' counters must be left at zero by every plan
    and never overlap another call's data."""
    import nvfp4_router_gate_gb300 as R
    base = WL.WORKLOADS["prefill"]
    ws = R.new_workspace(R.router_gate_workspace_size(4096, base.D, base.N, base.k))
    calls = []
    for T in (4096, 64, 1024, 4096, 2048, 256, 4096):
        case = Case(base.with_T(T))
        ids, wts = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, base.k,
                                      base.routed_scaling, base.raw, workspace=ws)
        calls.append((T, case, ids, wts, R.last_router_plan()))
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == 0
    for T, case, ids, wts, plan in calls:
        rows = np.unique(np.concatenate([np.arange(0, T, 97), [T - 1]]))
        res = case.check(ids.cpu().numpy(), wts.cpu().numpy(), rows)
        assert compare.topk_ok(res), (T, plan, res)


@pytest.mark.parametrize("flags", [DEC, TC])
def test_huge_logits_saturate_without_nan(flags):
    """x scaled by 2^10: logits reach +-3e4, every sigmoid saturates to 0 or 1
    (exp(-l) overflows for very negative logits; the scores must stay 0, not
    NaN) and the bias alone orders the saturated experts."""
    w = WL.WORKLOADS["decode"].with_T(8)
    case = Case(w)
    bits = WL.float32_to_bf16_bits((case.x32 * np.float32(1024.0)).astype(np.float32))
    import nvfp4_router_gate_gb300 as R
    ids, wts = R.router_gate_topk(to_device(bits, "bf16"), case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev,
                                  w.k, w.routed_scaling, w.raw, flags=flags)
    torch.cuda.synchronize()
    ids, wts = ids.cpu().numpy(), wts.cpu().numpy()
    assert np.all(np.isfinite(wts))
    x32 = WL.bf16_bits_to_float32(bits)
    gsa = Q.global_scale(x32)
    xq, xs, _ = Q.quantize(x32, gsa=gsa)
    L, B = gemm.logits(xq, xs, gsa, case.wq, case.ws, case.wg)
    keys = router.selection_keys(L, case.bias, w.raw)
    res = compare.check_topk(ids, wts, L, B, keys, case.bias, w.routed_scaling, w.raw)
    assert compare.topk_ok(res), res


# Decode calls of 3 or more tokens share the quantization of x across the
# grid (a barrier in the workspace between quantizing a slice and loading
# the rest); calls back to back on one workspace reuse the barrier.

@pytest.mark.parametrize("T", [3, 5, 7, 12, 16])
def test_decode_shared_quantization_ragged_token_counts(T):
    case = Case(WL.WORKLOADS["decode"].with_T(T))
    ids, w = case.run(DEC)
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res


def test_decode_shared_quantization_back_to_back_on_one_workspace():
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["decode"].with_T(8)
    case = Case(w)
    ws = R.new_workspace(R.router_gate_workspace_size(w.T, w.D, w.N, w.k))
    outs = []
    for scale in (1.0, 2.0 ** 10, 2.0 ** -12, 3.0, 1.0):
        bits = WL.float32_to_bf16_bits((case.x32 * np.float32(scale)).astype(np.float32))
        ids, wts = R.router_gate_topk(to_device(bits, "bf16"), case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev,
                                      w.k, w.routed_scaling, w.raw, workspace=ws, flags=DEC)
        outs.append((scale, bits, ids, wts))
    torch.cuda.synchronize()
    rows = np.arange(w.T)
    for scale, bits, ids, wts in outs:
        x32 = WL.bf16_bits_to_float32(bits)
        gsa = Q.global_scale(x32)
        xq, xs, _ = Q.quantize(x32, gsa=gsa)
        L, B = gemm.logits(xq, xs, gsa, case.wq, case.ws, case.wg)
        keys = router.selection_keys(L, case.bias, w.raw)
        res = compare.check_topk(ids.cpu().numpy(), wts.cpu().numpy(), L, B, keys, case.bias,
                                 w.routed_scaling, w.raw)
        assert compare.topk_ok(res), (scale, res)


# Decode calls of up to 256 experts: CTA 0 collects every (token, expert)
# key by polling words that each call leaves at zero (a fixed region of the
# workspace, clear of the regions whose place depends on T).  Calls of every
# decode shape, raw and biased, with a prefill call between them, on one
# workspace: a word left behind by one call would route the next wrongly.

def _oracle_check(case, x_bits, ids, wts, k, raw):
    x32 = WL.bf16_bits_to_float32(x_bits)
    gsa = Q.global_scale(x32)
    xq, xs, _ = Q.quantize(x32, gsa=gsa)
    L, B = gemm.logits(xq, xs, gsa, case.wq, case.ws, case.wg)
    keys = router.selection_keys(L, case.bias, raw)
    return compare.check_topk(ids, wts, L, B, keys, case.bias, case.w.routed_scaling, raw)


def test_decode_collector_words_across_calls_and_shapes():
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["decode"].with_T(16)
    case = Case(w)
    pre = WL.WORKLOADS["prefill"].with_T(600)
    x_pre = to_device(WL.make_x(pre), "bf16")
    ws = R.new_workspace(R.router_gate_workspace_size(600, w.D, w.N, 16))
    plan = [(1, 1.0, 8, False), (16, 2.0 ** 6, 8, False), (1, 3.0, 8, True), ("prefill", 0, 8, False),
            (1, 2.0 ** -9, 16, False), (8, 1.0, 1, False), (5, 0.5, 8, True), (1, 1.0, 8, False)]
    for T, scale, k, raw in plan:
        if T == "prefill":
            R.router_gate_topk(x_pre, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5, workspace=ws)
            continue
        bits = WL.float32_to_bf16_bits((case.x32[:T] * np.float32(scale)).astype(np.float32))
        ids, wts = R.router_gate_topk(to_device(bits, "bf16"), case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev,
                                      k, w.routed_scaling, raw, workspace=ws, flags=DEC)
        torch.cuda.synchronize()
        assert R.last_router_plan()["sequence"] == "decode"
        res = _oracle_check(case, bits, ids.cpu().numpy(), wts.cpu().numpy(), k, raw)
        assert compare.topk_ok(res), (T, scale, k, raw, res)
    assert R.nvr_read_device_status(ws) == 0


@pytest.mark.parametrize("T", [1, 8])
def test_decode_collector_timeout_reports_status(T):
    """Failure detection without a GPU fault: with the stall hook the decode
    CTAs other than the collector store no keys, the collector's poll runs
    out after about a second, records NVR_ERR_TIMEOUT and returns; after
    re-zeroing the workspace the next call routes correctly."""
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    case = Case(WL.WORKLOADS["decode"].with_T(T))
    ws = R.new_workspace(R.router_gate_workspace_size(T, 7168, 256, 8))
    R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                       workspace=ws, flags=DEC | _native.NVR_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == _native.NVR_ERR_TIMEOUT
    ws.zero_()
    ids, w = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                                workspace=ws, flags=DEC)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == 0
    res = case.check(ids.cpu().numpy(), w.cpu().numpy(), np.arange(T))
    assert compare.topk_ok(res), res


# ------------------------------------------------ quantization inside the GEMM
# bf16 activations on heads of up to 256 experts are quantized inside the GEMM
# kernel; the codes never reach memory.  A one-hot gate weight makes every
# logit a single product code_x * scale_x * gsa_x * (dequantized 1.0), so the
# logits expose the kernel's code and scale of each probed x element.

def _one_hot_gate(cols, D):
    W = np.zeros((len(cols), D), np.float32)
    W[np.arange(len(cols)), cols] = 1.0
    return W


def _fused_probe_x(rng, T, D):
    """bf16 rows: half with gsa = 1 and crafted blocks (E2M1 midpoints times
    each E4M3 significand, their bf16 neighbours, zeros, subnormals), half
    random with per-token LogNormal scale."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    x = (rng.standard_normal((T, D)) * np.exp(rng.standard_normal((T, 1)))).astype(np.float32)
    bits = WL.float32_to_bf16_bits(x)
    for t in range(T // 2):
        for b in range(D // 16):
            m, e = (t + b) % 8, (b % 5) - 2
            s = (8 + m) / 8.0 * 2.0 ** e
            vals = np.zeros(16, np.float32)
            vals[0] = 6.0 * s                                   # block scale exactly s
            probe = mids[(b + np.arange(15)) % 7] * s * rng.choice([-1, 1], 15)
            vals[1:] = probe
            vb = WL.float32_to_bf16_bits(vals)
            k = (t * 7 + b) % 4                                 # bf16 neighbours of the ties
            vb[1:8] = (vb[1:8].astype(np.int32) + [0, 1, -1, 2, -2, 0, k][:7]).astype(np.uint16)
            vb[8] = 0x8000 if b % 3 == 0 else 0x0001           # -0 or the smallest subnormal
            bits[t, 16 * b:16 * b + 16] = vb
    bits[0, 5] = WL.float32_to_bf16_bits(np.array([2688.0], np.float32))[0]   # gsa = 1 for the first half
    return bits


@pytest.mark.parametrize("flags", [0, K2, K8])
def test_fused_quantizer_codes_via_one_hot_gate(flags):
    import nvfp4_router_gate_gb300 as R
    rng = np.random.default_rng(31)
    T, D = 192, 512
    for half_x in range(2):
        bits = _fused_probe_x(rng, T, D)
        if half_x:                                     # the random half alone: arbitrary gsa
            bits = bits[T // 2:].copy()
        x32 = WL.bf16_bits_to_float32(bits)
        xd = to_device(bits, "bf16")
        xq, xs, xg = Q.quantize(x32)
        for c0 in range(0, D, 256):
            cols = np.arange(c0, c0 + 256)
            W = _one_hot_gate(cols, D)
            wf, wsf, wg = R.nvfp4_pack_weight(to_device(W, "f32"))
            out = R.router_gate_logits(xd, wf, wsf, wg, flags=flags)
            torch.cuda.synchronize()
            wq, wsb, wgg = Q.quantize(W)
            L, _ = gemm.logits(xq, xs, xg, wq, wsb, wgg)
            g = out.cpu().numpy().astype(np.float64)
            err = np.abs(g - L)
            assert np.all(err <= 1e-6 * np.abs(L)), (half_x, c0, np.argwhere(err > 1e-6 * np.abs(L))[:5])


def _probe_x_vectorized(rng, T, D, crafted):
    """_fused_probe_x for batches too large for a Python loop: the rows in the
    boolean mask `crafted` get the crafted blocks (E2M1 midpoints times every
    E4M3 significand and their bf16 neighbours, zeros, subnormals; gsa = 1 for
    the whole batch), the others LogNormal-scaled normals."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    x = (rng.standard_normal((T, D)) * np.exp(rng.standard_normal((T, 1)))).astype(np.float32)
    bits = WL.float32_to_bf16_bits(x)
    rows = np.nonzero(crafted)[0]
    nb = D // 16
    t = rows[:, None]
    b = np.arange(nb)[None, :]
    s = (8 + (t + b) % 8) / 8.0 * 2.0 ** ((b % 5) - 2)                  # block scale, [R, nb]
    vals = np.zeros((rows.size, nb, 16), np.float32)
    vals[:, :, 0] = 6.0 * s
    probe = mids[(b[..., None] + np.arange(15)) % 7]                  # [1, nb, 15]
    vals[:, :, 1:] = probe * s[..., None] * rng.choice([-1, 1], (rows.size, nb, 15))
    vb = WL.float32_to_bf16_bits(vals).astype(np.int32)
    off = np.zeros((rows.size, nb, 7), np.int32)
    off[:, :, :6] = [0, 1, -1, 2, -2, 0]                              # bf16 neighbours of the ties
    off[:, :, 6] = (t * 7 + b) % 4
    vb[:, :, 1:8] += off
    vb[:, :, 8] = np.where(b % 3 == 0, 0x8000, 0x0001)                # -0 or the smallest subnormal
    bits[rows] = vb.astype(np.uint16).reshape(rows.size, D)
    bits[rows[0], 5] = WL.float32_to_bf16_bits(np.array([2688.0], np.float32))[0]
    return bits


def test_fused_quantizer_codes_production_plan():
    """The one-hot probe of the in-GEMM quantizer at the prefill shape
    (T = 4096, D = 7168), so that it runs the default plan's tiles, K split
    and row assignment: every x element's code and scale byte is read back
    through one logit, on a batch with crafted rows (gsa = 1) and on a plain
    LogNormal batch (arbitrary gsa)."""
    import nvfp4_router_gate_gb300 as R
    rng = np.random.default_rng(41)
    T, D = 4096, 7168
    ws = R.new_workspace(R.router_gate_workspace_size(T, D, 256, 8))
    for crafted in (rng.random(T) < 0.5, None):
        if crafted is None:
            bits = WL.make_x(WL.WORKLOADS["prefill"])
        else:
            bits = _probe_x_vectorized(rng, T, D, crafted)
        x32 = WL.bf16_bits_to_float32(bits)
        xd = to_device(bits, "bf16")
        xq, xs, xg = Q.quantize(x32)
        if crafted is not None:
            assert xg == 1.0
        A = gemm.dequantize(xq, xs)
        plans = set()
        for c0 in range(0, D, 256):
            cols = np.arange(c0, c0 + 256)
            W = _one_hot_gate(cols, D)
            wf, wsf, wg = R.nvfp4_pack_weight(to_device(W, "f32"))
            out = R.router_gate_logits(xd, wf, wsf, wg, workspace=ws)
            plans.add(tuple(sorted(R.last_router_plan().items())))
            torch.cuda.synchronize()
            assert np.float32(R.router_gate_x_gsa(ws).item()) == xg
            wq, wsb, wgg = Q.quantize(W)
            wv = gemm.dequantize(wq, wsb)[np.arange(256), cols]        # the one nonzero of each row
            L = A[:, cols] * (wv * (np.float64(xg) * np.float64(wgg)))[None, :]
            g = out.cpu().numpy().astype(np.float64)
            err = np.abs(g - L)
            assert np.all(err <= 1e-6 * np.abs(L)), (c0, np.argwhere(err > 1e-6 * np.abs(L))[:5])
        assert len(plans) == 1 and dict(next(iter(plans)))["sequence"] == "fused", plans


def test_fused_router_next_to_kernels_holding_sms():
    """Half the SMs held by another stream's kernel (200 KB of shared memory
    each, released by itself after 20 ms) while the one-launch prefill router
    starts: its grid cannot all be resident until they return.  The call must
    complete with status OK and route like the oracle; a cooperative launch
    (when the runtime accepts it) waits for the whole grid, else the grid
    barrier's bounded wait absorbs the delay."""
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    w = WL.WORKLOADS["prefill"]
    case = Case(w)
    ws = R.new_workspace(R.router_gate_workspace_size(w.T, w.D, w.N, w.k))
    R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, w.k, w.routed_scaling,
                       workspace=ws)
    torch.cuda.synchronize()
    other = torch.cuda.Stream()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lib = _native.lib()
    for _ in range(2):
        _native.check("nvr_test_occupy",
                      lib.nvr_test_occupy(sms // 2, 200 * 1024, 20_000_000, ctypes_stream(other)))
        ids, wts = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, w.k,
                                      w.routed_scaling, workspace=ws)
        torch.cuda.synchronize()
        assert R.last_router_plan()["sequence"] == "fused"
        assert R.nvr_read_device_status(ws) == 0
        res = case.check(ids.cpu().numpy(), wts.cpu().numpy(), np.arange(w.T))
        assert compare.topk_ok(res), res
    assert lib.nvr_router_cooperative_state() in (1, -1)
    print("cooperative launch state:", lib.nvr_router_cooperative_state())


def ctypes_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)


def test_no_cooperative_flag_routes_identically():
    """NVR_FLAG_NO_COOPERATIVE changes only how the one-launch router is
    launched: ids and weights are bit-identical to the default call's."""
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS["prefill"]
    case = Case(w.with_T(2048))
    a_ids, a_w = case.run(0)
    b_ids, b_w = case.run(R.NVR_FLAG_NO_COOPERATIVE)
    assert R.last_router_plan()["sequence"] == "fused"
    assert np.array_equal(a_ids, b_ids) and np.array_equal(a_w.view(np.uint32), b_w.view(np.uint32))


@pytest.mark.parametrize("N", [300, 384])
@pytest.mark.parametrize("T", [8, 200])
def test_exact_integer_logits_up_to_384_experts(N, T):
    """The one-launch kernel for heads of 257-384 experts (two MMAs per K
    step, N = 256 and N = 128, into 384 accumulator columns): grid-valued
    operands give exact logits (any fp32 summation order), so the GPU must
    equal the oracle's bits, the ragged last group included."""
    import nvfp4_router_gate_gb300 as R
    rng = np.random.default_rng(23)
    D = 512
    x = _grid_operands(rng, T, D, 0)
    W = _grid_operands(rng, N, D, 1)
    wf, ws, wg = R.nvfp4_pack_weight(to_device(W, "f32"))
    xd = to_device(x, "f32").to(torch.bfloat16)        # the one-launch kernel takes bf16 x
    assert torch.equal(xd.float().cpu(), torch.from_numpy(x))   # grid values are bf16-exact
    out = R.router_gate_logits(xd, wf, ws, wg, flags=TC)
    torch.cuda.synchronize()
    assert R.last_router_plan()["sequence"] in ("fused", "amax+fused")
    xq, xs, xg = Q.quantize(x)
    wq, wsb, wgg = Q.quantize(W)
    L, _ = gemm.logits(xq, xs, xg, wq, wsb, wgg)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), L)


@pytest.mark.parametrize("N,T,k,raw", [(384, 129, 8, False), (300, 300, 16, False), (384, 2048, 8, False),
                                       (384, 300, 1, True), (320, 40, 8, False)])
def test_router_up_to_384_experts_all_rows(N, T, k, raw):
    """Every row of prefill-like batches on heads of 257-384 experts through
    the one-launch kernel (its plans: clusters of up to 16 CTAs, or 8 CTAs per
    tile without clusters at T = 2048)."""
    import nvfp4_router_gate_gb300 as R
    w = WL.Workload("wide_gate", T, 7168, N, k, 1.0 if raw else 2.5, raw, "bf16", "lognormal_rows", 0.02,
                    "uniform", 0.05)
    case = Case(w)
    ids, wts = case.run()
    assert R.last_router_plan()["sequence"] == "fused"
    res = case.check(ids, wts, np.arange(T))
    assert compare.topk_ok(res), res


def test_router_384_experts_two_launch_plan():
    """More token tiles than the GPU holds at once (T = 20000: 157 tiles of
    128 rows > 152 CTAs): the amax kernel, then the fused kernel for 384
    experts reading its record; every row against the oracle."""
    import nvfp4_router_gate_gb300 as R
    w = WL.Workload("wide_gate_large", 20000, 7168, 384, 8, 2.5, False, "bf16", "lognormal_rows", 0.02,
                    "uniform", 0.05)
    case = Case(w)
    ids, wts = case.run()
    assert R.last_router_plan()["sequence"] == "amax+fused", R.last_router_plan()
    res = case.check(ids, wts, np.arange(w.T))
    assert compare.topk_ok(res), res
