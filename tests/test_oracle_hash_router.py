"""Pins of the hash-router oracle (oracle/hash_router.py): a worked case
written out by hand (tests/golden/hash_router_case.txt), and the plain
properties of a lookup on the seeded workload."""

import os

import numpy as np

import workloads as WL
from oracle import hash_router

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hash_router_case.txt")


def _read_case():
    rows = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, vals = line.split(":")
        rows[key.strip()] = vals.split()
    table = np.array([[int(v) for v in rows["table %d" % i]] for i in range(4)], np.int32)
    tokens = np.array([int(v) for v in rows["tokens"]], np.int64)
    ids = np.array([[int(v) for v in rows["ids %d" % t]] for t in range(len(tokens))], np.int32)
    w = np.array([[int(v, 16) if v.startswith("0x") else int(v) for v in rows["weights %d" % t]]
                  for t in range(len(tokens))], np.uint32).view(np.float32)
    return table, tokens, ids, w


def test_hash_router_worked_case():
    table, tokens, ids, w = _read_case()
    got_ids, got_w = hash_router.route(tokens, table, 10, 1.0)
    assert np.array_equal(got_ids, ids)
    assert np.array_equal(got_w.view(np.uint32), w.view(np.uint32))
    assert got_w[0, 0] == np.float32(1.0) / np.float32(3.0)


def test_hash_router_workload_properties():
    hw = WL.HASH_ROUTER
    table = WL.make_hash_table(hw)
    tids = WL.make_token_ids(hw)
    assert table.shape == (hw.vocab, hw.k) and table.dtype == np.int32
    assert np.all((table >= 0) & (table < hw.n_experts))
    assert all(len(set(r)) == hw.k for r in table[:1000].tolist())         # distinct experts per token
    ids, w = hash_router.route(tids[:300], table, hw.n_experts, hw.routed_scaling)
    assert np.array_equal(ids, table[tids[:300]])                           # a pure gather
    assert np.all(w == np.float32(hw.routed_scaling / hw.k))
    assert np.allclose(w.sum(axis=1), hw.routed_scaling)
