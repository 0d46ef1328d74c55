"""GPU parity of the NVFP4 grouped expert GEMM (nvfp4_moe_gemm) and the
weighted combine (nvfp4_moe_combine) against the oracle (oracle/moe.py):
random routing, skewed routing (an expert with several 128-row token tiles,
empty experts, out-of-range ids), fp32 and bf16 outputs, the router's own
ids fed straight in, and CUDA-graph replay."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from oracle import quantize as Q, moe, compare  # noqa: E402
from gpu_util import to_device  # noqa: E402


def _experts(rng, E, N, D, dtype="bf16"):
    W = (rng.standard_normal((E, N, D)) * 0.02).astype(np.float32)
    if dtype == "bf16":
        bits = WL.float32_to_bf16_bits(W)
        return bits, WL.bf16_bits_to_float32(bits)
    return W, W


def _run(x_bits, x32, ids, Wdev, W32, dt="bf16", out="f32", w=None):
    import nvfp4_router_gate_gb300 as R
    wf, wsf, wg = R.nvfp4_pack_experts(Wdev)
    xd = to_device(x_bits, dt)
    idd = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    y = R.nvfp4_moe_gemm(xd, idd, wf, wsf, wg, out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    comb = None
    if w is not None:
        comb = R.nvfp4_moe_combine(y, torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda())
    torch.cuda.synchronize()
    packed = [Q.quantize(W32[e]) for e in range(W32.shape[0])]
    # the experts' global scales must be the oracle's bits
    assert np.array_equal(wg.cpu().numpy().view(np.uint32), np.array([p[2] for p in packed], np.float32).view(np.uint32))
    return y.float().cpu().numpy(), None if comb is None else comb.cpu().numpy(), packed


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_moe_random_routing(out):
    rng = np.random.default_rng(51)
    T, D, E, N, k = 96, 512, 8, 256, 2
    x = (rng.standard_normal((T, D)) * np.exp(rng.standard_normal((T, 1)))).astype(np.float32)
    xb = WL.float32_to_bf16_bits(x)
    x32 = WL.bf16_bits_to_float32(xb)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    Wb, W32 = _experts(rng, E, N, D)
    w = rng.random((T, k)).astype(np.float32)
    y, comb, packed = _run(xb, x32, ids, to_device(Wb.reshape(E * N, D), "bf16").view(E, N, D), W32, out=out, w=w)
    Y, B = moe.grouped_gemm(x32, ids, packed)
    if out == "f32":
        assert compare.check_logits(y.reshape(T * k, N), Y.reshape(T * k, N), B.reshape(T * k, N)) == 0
        assert compare.check_moe_combine(comb, Y, B, w) == 0
    else:
        assert compare.check_logits_bf16(y.reshape(T * k, N), Y.reshape(T * k, N), B.reshape(T * k, N)) == 0


def test_moe_skewed_routing_and_bad_ids():
    """Most pairs on expert 0 (several 128-row token tiles), experts 4..7 with
    no rows, ids -1 and E (zero output rows); fp32 activations."""
    rng = np.random.default_rng(52)
    T, D, E, N, k = 300, 256, 8, 128, 2
    x = rng.standard_normal((T, D)).astype(np.float32)
    ids = np.zeros((T, k), np.int32)
    ids[:, 1] = rng.integers(1, 4, T)
    ids[5, 1] = -1
    ids[17, 0] = E
    Wf, W32 = _experts(rng, E, N, D, dtype="f32")
    y, _, packed = _run(x, x, ids, to_device(Wf.reshape(E * N, D), "f32").view(E, N, D), W32, dt="f32")
    valid = (ids >= 0) & (ids < E)
    Y, B = moe.grouped_gemm(x, np.where(valid, ids, 0), packed)
    ok = valid.ravel()
    assert compare.check_logits(y.reshape(T * k, N)[ok], Y.reshape(T * k, N)[ok], B.reshape(T * k, N)[ok]) == 0
    assert np.all(y[~valid] == 0.0)


def test_moe_fed_by_the_router():
    """The router's ids and weights (E = 16 experts, k = 4, T = 200 prefill
    rows, D = 7168) straight into the grouped GEMM and the combine."""
    import nvfp4_router_gate_gb300 as R
    from gpu_util import Case
    gw = WL.Workload("moe_gate", 200, 7168, 16, 4, 2.5, False, "bf16", "lognormal_rows", 0.02, "uniform", 0.05)
    case = Case(gw)
    ids_d, w_d = R.router_gate_topk(case.x_dev, case.W_fp4, case.W_sf, case.w_gsa, case.bias_dev, gw.k,
                                    gw.routed_scaling)
    rng = np.random.default_rng(53)
    E, N = 16, 128
    Wb, W32 = _experts(rng, E, N, gw.D)
    wf, wsf, wg = R.nvfp4_pack_experts(to_device(Wb.reshape(E * N, gw.D), "bf16").view(E, N, gw.D))
    y = R.nvfp4_moe_gemm(case.x_dev, ids_d, wf, wsf, wg)
    out = R.nvfp4_moe_combine(y, w_d)
    torch.cuda.synchronize()
    ids, w = ids_d.cpu().numpy(), w_d.cpu().numpy()
    packed = [Q.quantize(W32[e]) for e in range(E)]
    Y, B = moe.grouped_gemm(case.x32, ids, packed)
    assert compare.check_logits(y.cpu().numpy().reshape(-1, N), Y.reshape(-1, N), B.reshape(-1, N)) == 0
    assert compare.check_moe_combine(out.cpu().numpy(), Y, B, w) == 0


def test_moe_graph_replay_without_sync_or_allocation():
    import nvfp4_router_gate_gb300 as R
    rng = np.random.default_rng(54)
    T, D, E, N, k = 64, 512, 4, 128, 2
    x = rng.standard_normal((T, D)).astype(np.float32)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    Wf, W32 = _experts(rng, E, N, D, dtype="f32")
    wf, wsf, wg = R.nvfp4_pack_experts(to_device(Wf.reshape(E * N, D), "f32").view(E, N, D))
    xd = to_device(x, "f32")
    idd = torch.from_numpy(ids).cuda()
    wd = torch.from_numpy(rng.random((T, k)).astype(np.float32)).cuda()
    ws = R.new_workspace(R.nvfp4_moe_gemm_workspace_size(T, D, E, k))
    y = torch.empty((T, k, N), dtype=torch.float32, device="cuda")
    out = torch.empty((T, N), dtype=torch.float32, device="cuda")
    R.nvfp4_moe_gemm(xd, idd, wf, wsf, wg, y=y, workspace=ws)
    R.nvfp4_moe_combine(y, wd, out=out)
    ref = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        R.nvfp4_moe_gemm(xd, idd, wf, wsf, wg, y=y, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        R.nvfp4_moe_gemm(xd, idd, wf, wsf, wg, y=y, workspace=ws)
        R.nvfp4_moe_combine(y, wd, out=out)
    out.zero_()
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.cuda.memory_allocated() == before
    assert R.nvr_read_device_status(ws) == 0
