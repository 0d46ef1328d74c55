"""GPU parity of the weight-streaming kernel (up to 128 tokens; weight rows as
the MMA's M, tokens as its N) against the oracle, through the C ABI: exact
integer logits, logits within tolerance for every token tile (32, 64, 128
columns), the router's top-k on heads of 256 and 384 experts (k = 1 to 16,
ties, RAW), the per-CTA list merge, and the NVFP4 linear (nvfp4_linear, fp32
and bf16 output; the N-split kernel for more than 128 tokens)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from oracle import quantize as Q, gemm, compare  # noqa: E402
from gpu_util import Case, to_device  # noqa: E402

ST = 128     # NVR_FLAG_STREAM


def _plan():
    import nvfp4_router_gate_gb300 as R
    return R.last_router_plan()


@pytest.mark.parametrize("T", [8, 40, 100])
def test_stream_exact_integer_logits(T):
    """Grid-valued operands (gsa = 1, power-of-two block scales): any fp32
    summation order is exact, so the logits must equal the oracle's bits --
    this pins the token tile's scale-factor layout for 32, 64 and 128 MMA
    columns."""
    import nvfp4_router_gate_gb300 as R
    from test_gpu_router import _grid_operands
    rng = np.random.default_rng(23)
    N, D = 392, 512
    x = _grid_operands(rng, T, D, 0)
    W = _grid_operands(rng, N, D, 1)
    wf, ws, wg = R.nvfp4_pack_weight(to_device(W, "f32"))
    out = R.router_gate_logits(to_device(x, "f32"), wf, ws, wg, flags=ST)
    torch.cuda.synchronize()
    assert _plan()["sequence"] == "amax+quantize+stream"
    xq, xs, xg = Q.quantize(x)
    wq, wsb, wgg = Q.quantize(W)
    L, _ = gemm.logits(xq, xs, xg, wq, wsb, wgg)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), L)


@pytest.mark.parametrize("name,T", [("decode", 1), ("decode", 8), ("prefill", 33), ("prefill", 64),
                                    ("prefill", 65), ("prefill", 128), ("adversarial", 96)])
def test_stream_logits_within_tolerance(name, T):
    import nvfp4_router_gate_gb300 as R
    case = Case(WL.WORKLOADS[name].with_T(T))
    out = R.router_gate_logits(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, flags=ST)
    torch.cuda.synchronize()
    L, B = case.oracle_rows(np.arange(T))
    assert compare.check_logits(out.cpu().numpy(), L, B) == 0


@pytest.mark.parametrize("T", [1, 8, 31, 64, 128])
@pytest.mark.parametrize("k", [1, 3, 8, 16])
def test_stream_router_256(T, k):
    case = Case(WL.WORKLOADS["decode"].with_T(T).with_k(k))
    ids, w = case.run(ST)
    assert _plan()["sequence"] == "amax+quantize+stream"
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res


@pytest.mark.parametrize("T", [16, 64, 100])
@pytest.mark.parametrize("flags", [0, ST])
def test_wide_head_adversarial_small_batches(T, flags):
    """The adversarial rows (all-zero rows tie every key at 0.5: ids 0..7;
    1e4 rows saturate) on E = 384 at up to 128 tokens: by default the decode
    kernel (T <= 16) or the one-launch kernel, forced the streaming kernel."""
    case = Case(WL.WORKLOADS["adversarial"].with_T(T))
    ids, w = case.run(flags)
    want = "amax+quantize+stream" if flags else ("decode" if T <= 16 else "fused")
    assert _plan()["sequence"] == want, _plan()
    res = case.check(ids, w, np.arange(T))
    assert compare.topk_ok(res), res
    zero = np.arange(1, T, 4)
    assert np.all(ids[zero] == np.arange(8))
    assert np.allclose(w[zero], 2.5 / 8, atol=1e-6)


def test_stream_router_ties_and_raw():
    w = WL.Workload("tie_probe_s", 96, 7168, 384, 8, 2.5, False, "bf16", "adversarial", 0.02, "zero",
                    tie_probe=True)
    case = Case(w)
    ids, wt = case.run(ST)
    res = case.check(ids, wt, np.arange(96))
    assert compare.topk_ok(res), res
    for row in ids:
        pos = {int(e): i for i, e in enumerate(row)}
        for e, i in pos.items():
            if e < 16 and e % 2 == 1 and (e - 1) in pos:
                assert pos[e - 1] < i
    w = WL.Workload("raw_600", 50, 7168, 600, 8, 1.0, True, "bf16", "normal", 0.02, "none")
    case = Case(w)
    ids, wt = case.run(ST)
    res = case.check(ids, wt, np.arange(50))
    assert compare.topk_ok(res), res


def test_stream_timeout_reports_status():
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    case = Case(WL.WORKLOADS["decode"].with_T(8))
    ws = R.new_workspace(R.router_gate_workspace_size(8, 7168, 256, 8))
    R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5, workspace=ws,
                       flags=ST | _native.NVR_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == _native.NVR_ERR_TIMEOUT
    ws.zero_()
    ids, w = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, 8, 2.5,
                                workspace=ws, flags=ST)
    torch.cuda.synchronize()
    assert R.nvr_read_device_status(ws) == 0
    res = case.check(ids.cpu().numpy(), w.cpu().numpy(), np.arange(8))
    assert compare.topk_ok(res), res


# ---------------------------------------------------------------- NVFP4 linear

@pytest.mark.parametrize("T,N", [(1, 2048), (32, 1000), (100, 4096), (128, 256), (300, 1536), (1000, 2048)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_nvfp4_linear(T, N, out_dtype):
    import nvfp4_router_gate_gb300 as R
    w = WL.Workload("linear", T, 7168, N, 1, 1.0, True, "bf16", "lognormal_rows", 0.02, "none")
    case = Case(w)
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = R.nvfp4_linear(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, out_dtype=dt)
    torch.cuda.synchronize()
    assert _plan()["sequence"] == ("amax+quantize+stream" if T <= 128 else "amax+quantize+splitn")
    L, B = case.oracle_rows(np.arange(T))
    g = out.float().cpu().numpy()
    if out_dtype == "f32":
        assert compare.check_logits(g, L, B) == 0
    else:
        assert compare.check_logits_bf16(g, L, B) == 0


def test_nvfp4_linear_resident_layer_graph_replay():
    """Nvfp4Linear: packed weight, workspace and output resident; a captured
    call replays to the same output (fp32 activations, the lm_head-like
    N = 129280 is left to the bench)."""
    import nvfp4_router_gate_gb300 as R
    w = WL.Workload("linear_g", 16, 1024, 3000, 1, 1.0, True, "f32", "normal", 0.05, "none")
    case = Case(w)
    lin = R.Nvfp4Linear(case.W_dev, max_tokens=16)
    ref = lin(case.x_dev).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lin(case.x_dev)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lin(case.x_dev)
    lin.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lin.out[:16], ref)
    L, B = case.oracle_rows(np.arange(16))
    assert compare.check_logits(ref.cpu().numpy(), L, B) == 0
