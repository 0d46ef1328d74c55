"""GPU parity of the hash router (router_hash_topk) against the oracle's
lookup: ids and weights bit-exact on the seeded workload (T = 4096, vocab =
129280, 256 experts, k = 8), ragged and empty batches, k = 1, out-of-range
token ids and table entries, and CUDA-graph replay."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from oracle import hash_router  # noqa: E402


def _run(tids, table, n_experts, rs):
    import nvfp4_router_gate_gb300 as R
    ids, w = R.router_hash_topk(torch.from_numpy(tids).cuda(), torch.from_numpy(table).cuda(), n_experts, rs)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _exact(got, want):
    gi, gw = got
    wi, ww = want
    assert np.array_equal(gi, wi)
    assert np.array_equal(gw.view(np.uint32), ww.view(np.uint32))


@pytest.mark.parametrize("T", [4096, 1, 777])
def test_hash_router_workload(T):
    h = WL.HASH_ROUTER.with_T(T)
    table = WL.make_hash_table(h)
    tids = WL.make_token_ids(h)
    _exact(_run(tids, table, h.n_experts, h.routed_scaling),
           hash_router.route(tids, table, h.n_experts, h.routed_scaling))


def test_hash_router_k1_and_out_of_range_inputs():
    rng = np.random.default_rng(3)
    table = rng.integers(-3, 12, (50, 1)).astype(np.int32)          # some entries outside [0, 10)
    tids = rng.integers(-5, 60, 333).astype(np.int32)               # some ids outside the table
    _exact(_run(tids, table, 10, 1.5), hash_router.route(tids, table, 10, 1.5))
    table = rng.integers(-3, 12, (50, 3)).astype(np.int32)
    _exact(_run(tids, table, 10, 1.0), hash_router.route(tids, table, 10, 1.0))


def test_hash_router_empty_batch_and_errors():
    import nvfp4_router_gate_gb300 as R
    table = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    ids, w = R.router_hash_topk(torch.zeros(0, dtype=torch.int32, device="cuda"), table, 4, 1.0)
    assert ids.shape == (0, 2)
    with pytest.raises(R.RouterError):
        R.router_hash_topk(torch.zeros(3, dtype=torch.int32, device="cuda"), table, 1, 1.0)   # k > n_experts


def test_hash_router_graph_replay():
    import nvfp4_router_gate_gb300 as R
    h = WL.HASH_ROUTER
    table = torch.from_numpy(WL.make_hash_table(h)).cuda()
    tids_np = WL.make_token_ids(h)
    tids = torch.from_numpy(tids_np).cuda()
    ids = torch.empty((h.T, h.k), dtype=torch.int32, device="cuda")
    w = torch.empty((h.T, h.k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        R.router_hash_topk(tids, table, h.n_experts, h.routed_scaling, ids, w)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        R.router_hash_topk(tids, table, h.n_experts, h.routed_scaling, ids, w)
    ids.zero_()
    g.replay()
    torch.cuda.synchronize()
    _exact((ids.cpu().numpy(), w.cpu().numpy()), hash_router.route(tids_np, table.cpu().numpy(), h.n_experts,
                                                                  h.routed_scaling))
