"""The router's launch planner on the host (no GPU): the plan query runs the
same function the dispatch runs, here with the capacities of a 152-SM device
whose GPCs hold whole clusters only (fewer CTAs in clusters than without)."""

import os
import shutil

import pytest

from nvfp4_router_gate_gb300 import _native

D, N = 7168, 256
SMS = 152
CAPS = (152, 76, 32, 16, 6)      # clusters of 1, 2, 4, 8, 16 CTAs held at once
BLOCKS = 152                     # CTAs held at once without clusters


def _lib():
    from nvfp4_router_gate_gb300 import build
    if not os.path.exists(_native.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("library not built and no nvcc")
        build.build()
    return _native.lib()


def plan(T, n=N, dtype="bf16", flags=0, caps=CAPS, blocks=BLOCKS):
    _lib()
    import nvfp4_router_gate_gb300 as R
    return R.plan_router(T, D, n, num_sms=SMS, cluster_capacity=caps, block_capacity=blocks, dtype=dtype,
                         flags=flags)


@pytest.mark.parametrize("T,expect", [
    (4096, ("fused", 112, 4, False)),     # 37 x 4 = 148 CTAs without clusters; clusters of 4 hold 32 tiles
    (3001, ("fused", 112, 4, True)),      # 27 tiles fit in clusters: clusters win the tie
    (2048, ("fused", 112, 8, False)),     # 19 x 8 = 152 CTAs
    (1024, ("fused", 128, 16, False)),    # 8 clusters of 16 do not fit, 128 CTAs do
    (512, ("fused", 112, 16, True)),
    (256, ("fused", 112, 16, True)),
    (64, ("fused", 112, 16, True)),       # one cluster
    (17, ("fused", 112, 16, True)),
])
def test_prefill_plans(T, expect):
    p = plan(T)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"], p["clustered"]) == expect, p


def test_decode_plans():
    assert plan(1)["sequence"] == "decode" and not plan(1)["clustered"]
    for T in (2, 8, 16):
        p = plan(T)
        assert p["sequence"] == "decode" and p["clustered"], (T, p)
    # forced tensor cores take the fused kernel even for one token
    assert plan(1, flags=_native.NVR_FLAG_FORCE_TENSOR_CORE)["sequence"] == "fused"
    # a forced decode of a batch too large for it is refused
    with pytest.raises(Exception):
        plan(64, flags=_native.NVR_FLAG_FORCE_DECODE)


def test_other_sequences():
    p = plan(4096, dtype="f32")
    assert p["sequence"] == "amax+quantize+splitk+epilogue" and p["ctas_per_tile"] == 4, p
    # 257-384 experts with bf16 x: the one-launch kernel too (147 tiles of 112
    # rows, one CTA each, all resident); fp32 x keeps the N-split path
    p = plan(16384, n=384)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"]) == ("fused", 112, 1), p
    p = plan(16384, n=384, dtype="f32")
    assert p["sequence"] == "amax+quantize+splitn" and p["tile_rows"] == 128, p
    p = plan(4096, flags=_native.NVR_FLAG_SPLIT_N)
    assert p["sequence"] == "amax+quantize+splitn", p
    # wide heads at up to 128 tokens stream the weight: token tiles of 32, 64
    # or 128 MMA columns, one CTA per SM (at most one per 128-row weight tile)
    for T, tn in ((1, 32), (32, 32), (33, 64), (64, 64), (65, 128), (128, 128)):
        p = plan(T, n=129280)
        assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"]) == ("amax+quantize+stream", tn, SMS), (T, p)
    assert plan(129, n=129280)["sequence"] == "amax+quantize+splitn"
    p = plan(40, n=384)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"]) == ("fused", 112, 16), p
    p = plan(40, n=384, flags=_native.NVR_FLAG_STREAM)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"]) == ("amax+quantize+stream", 64, 3), p
    assert plan(40, n=385)["sequence"] == "amax+quantize+stream"
    p = plan(100, flags=_native.NVR_FLAG_STREAM)
    assert (p["sequence"], p["ctas_per_tile"]) == ("amax+quantize+stream", 2), p
    assert plan(32, n=129280, flags=_native.NVR_FLAG_SPLIT_N)["sequence"] == "amax+quantize+splitn"
    with pytest.raises(Exception):
        plan(200, flags=_native.NVR_FLAG_STREAM)            # more tokens than one token tile
    # a forced split keeps 128-row tiles; 20 clusters of 8 are not resident at
    # once, so the amax kernel runs first
    p = plan(2560, flags=_native.NVR_FLAG_SPLIT_K_8)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"], p["clustered"]) == ("amax+fused", 128, 8, True), p
    p = plan(2560, flags=_native.NVR_FLAG_SPLIT_K_2)
    assert (p["sequence"], p["tile_rows"], p["ctas_per_tile"]) == ("fused", 128, 2), p
    # more tiles than the device holds: two launches
    assert plan(40000)["sequence"] == "amax+fused"


def test_one_launch_plans_are_resident_and_cheapest():
    """Every one-launch plan fits the device at once, and no resident
    alternative does less work per CTA (rows x K stages)."""
    n_st = (D // 16 + 15) // 16
    for T in list(range(17, 600, 7)) + list(range(600, 20000, 397)):
        p = plan(T)
        assert p["sequence"] in ("fused", "amax+fused"), (T, p)
        if p["sequence"] != "fused":
            continue
        rows, S = p["tile_rows"], p["ctas_per_tile"]
        tiles = -(-T // rows)
        if p["clustered"]:
            assert CAPS[S.bit_length() - 1] >= tiles, (T, p)
        else:
            assert tiles * S <= BLOCKS, (T, p)
        cost = rows * (-(-n_st // S))
        for r in (128, 112):
            t = -(-T // r)
            for c in (1, 2, 4, 8, 16):
                fits = CAPS[c.bit_length() - 1] >= t or (c > 1 and t * c <= BLOCKS)
                if fits and c <= S_max(T):
                    assert r * (-(-n_st // c)) >= cost, (T, p, r, c)


def S_max(T):
    """The most K splits the planner may use for T tokens: SMs per 128-row
    tile, at most 16 and the K stages, and what the workspace's partial
    region holds (16 planes of the padded batch, or 256 tiles' worth)."""
    m_tiles = -(-T // 128)
    s = max(1, min(SMS // m_tiles, 16, (D // 16 + 15) // 16))
    cap = min(16 * m_tiles * 128, max(m_tiles * 128, 256 * 128)) // (m_tiles * 128)
    return min(s, cap)


def test_plan_query_rejects_bad_arguments():
    import ctypes
    L = _lib()
    caps = (ctypes.c_int * 5)(*CAPS)
    out = (ctypes.c_int * 4)()
    ok = L.nvr_plan_router(4096, D, N, _native.NVR_BF16, 0, SMS, caps, BLOCKS, out)
    assert ok == _native.NVR_OK
    bad = [
        (0, D, N, _native.NVR_BF16, 0, SMS, caps, BLOCKS, out),            # T < 1
        (64, 200, N, _native.NVR_BF16, 0, SMS, caps, BLOCKS, out),         # D % 64
        (64, D, 0, _native.NVR_BF16, 0, SMS, caps, BLOCKS, out),           # N < 1
        (64, D, N, 7, 0, SMS, caps, BLOCKS, out),                          # dtype
        (64, D, N, _native.NVR_BF16, 512, SMS, caps, BLOCKS, out),         # unknown flag
        (64, D, N, _native.NVR_BF16, _native.NVR_FLAG_FORCE_DECODE | _native.NVR_FLAG_FORCE_TENSOR_CORE,
         SMS, caps, BLOCKS, out),
        (64, D, N, _native.NVR_BF16, 0, 0, caps, BLOCKS, out),             # no SMs
        (64, D, N, _native.NVR_BF16, 0, SMS, None, BLOCKS, out),
        (64, D, N, _native.NVR_BF16, 0, SMS, caps, BLOCKS, None),
    ]
    for args in bad:
        assert L.nvr_plan_router(*args) == _native.NVR_ERR_INVALID_ARG, args
    assert L.nvr_plan_router(64, D, 384, _native.NVR_BF16, _native.NVR_FLAG_SPLIT_K_4, SMS, caps, BLOCKS,
                             out) == _native.NVR_ERR_UNSUPPORTED


def test_tiny_fp32_router_is_one_launch():
    """The fp32 tiny router (T = 4, D = 256, E = 16) runs the single-launch
    decode kernel: one launch for fp32 activations too, at decode sizes."""
    _lib()
    import nvfp4_router_gate_gb300 as R
    p = R.plan_router(4, 256, 16, num_sms=SMS, cluster_capacity=CAPS, block_capacity=BLOCKS, dtype="f32", flags=0)
    assert p["sequence"] == "decode", p
