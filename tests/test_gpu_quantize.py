"""GPU parity of the quantize kernels against the oracle: bit-exact gsa, codes
and scale bytes, on the seeded workloads and on crafted inputs that sit on the
E2M1 / E4M3 rounding boundaries, on the division shortcut's range limits and
on the degenerate tensors (all zero, subnormal, tiny and huge magnitudes)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from oracle import formats, quantize as Q  # noqa: E402
from gpu_util import to_device, as_f32, f32_bits  # noqa: E402


def _gpu_quant(x_dev, layout):
    import nvfp4_router_gate_gb300 as R
    c, s, g = R.nvfp4_quantize_act(x_dev, sf_layout=layout)
    torch.cuda.synchronize()
    return c.cpu().numpy(), s.cpu().numpy(), g.cpu().numpy()[0]


def _check_exact(x32, x_dev, layout="linear"):
    codes, sf, gsa = _gpu_quant(x_dev, layout)
    q, sb, g = Q.quantize(x32)
    assert f32_bits(gsa) == f32_bits(g), (gsa, g)
    exp_codes = Q.pack_fp4(q)
    bad = np.nonzero(codes != exp_codes)
    assert bad[0].size == 0, "codes differ at %s: gpu %s oracle %s" % (
        list(zip(*bad))[:5], codes[bad][:5], exp_codes[bad][:5])
    if layout == "linear":
        assert np.array_equal(sf.reshape(sb.shape), sb)
    else:
        assert np.array_equal(sf, Q.sf_to_tiles(sb))


@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode", 1), ("decode", 8), ("decode", 64),
                                    ("prefill", 300), ("adversarial", 64)])
@pytest.mark.parametrize("layout", ["linear", "tiled"])
def test_quantize_workloads(name, T, layout):
    w = WL.WORKLOADS[name].with_T(T)
    x = WL.make_x(w)
    _check_exact(as_f32(x, w.dtype), to_device(x, w.dtype), layout)


def test_quantize_full_prefill_batch():
    w = WL.WORKLOADS["prefill"]
    x = WL.make_x(w)
    _check_exact(as_f32(x, w.dtype), to_device(x, w.dtype), "tiled")


def _probe_block_rows(values, lead=6.0):
    """Rows of 16-element blocks: a leading `lead` and 15 probe values each."""
    v = np.asarray(values, np.float32)
    nb = (v.size + 14) // 15
    blocks = np.zeros((nb, 16), np.float32)
    blocks[:, 0] = lead
    flat = blocks[:, 1:].reshape(-1)
    flat[: v.size] = v
    blocks[:, 1:] = flat.reshape(nb, 15)
    nblk = ((nb + 3) // 4) * 4                       # whole 64-element rows
    out = np.zeros((nblk, 16), np.float32)
    out[:nb] = blocks
    out[nb:, 0] = lead
    return out.reshape(-1, 64)


def test_e2m1_rounding_boundaries():
    """gsa = 1 exactly (amax 2688) and block scale 1 (block max 6): y/s = x."""
    grid = formats.E2M1_MAGNITUDES
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([grid, mids, [6.5, 7.0, 100.0, 1e-30, 1e-45]]).astype(np.float32)
    probes = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)),
                             np.nextafter(pts, np.float32(0))]).astype(np.float32)
    probes = np.concatenate([probes, -probes, [np.float32(-0.0)]]).astype(np.float32)
    probes = probes[np.abs(probes) <= 6.0]           # keep the block scale at exactly 1
    rows = _probe_block_rows(probes)
    rows[0, 0] = 2688.0                              # amax -> gsa = 1
    rows[0, 1:16] = 0.0
    _check_exact(rows, to_device(rows, "f32"))


def test_e2m1_boundaries_under_every_scale_mantissa():
    """y / s next to every E2M1 midpoint for block scales with each of the
    eight E4M3 significands (s = (8 + m) / 8 * 2^e): the quotient's last bit
    decides the code, which pins the one-correction division by s."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rows = []
    for e in (-3, 0, 2):
        for m in range(8):
            s = np.float32((8 + m) / 8.0 * 2.0 ** e)
            base = (mids.astype(np.float64) * float(s)).astype(np.float32)     # exact (<= 7 bits)
            probes = [base]
            for d in (1, 2, 3):
                up, dn = base.copy(), base.copy()
                for _ in range(d):
                    up = np.nextafter(up, np.float32(np.inf))
                    dn = np.nextafter(dn, np.float32(0))
                probes += [up, dn]
            p = np.concatenate(probes).astype(np.float32)
            p = np.concatenate([p, -p])
            blocks = _probe_block_rows(p, lead=np.float32(6.0) * s)
            rows.append(blocks)
    x = np.concatenate(rows)
    amax_row = np.zeros((4, 64), np.float32)
    amax_row[0, 0] = 2688.0                           # gsa = 1 (bigger than every lead)
    x = np.concatenate([amax_row, x]).astype(np.float32)
    _check_exact(x, to_device(x, "f32"))


def test_e4m3_rounding_boundaries():
    """Block maxima whose sy = max/6 lands on and next to every E4M3 midpoint."""
    vals = formats.E4M3_TABLE[:0x7F]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    targets = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                              np.nextafter(mids, np.float32(0)), vals.astype(np.float32),
                              [np.float32(2.0 ** -10), np.float32(2.0 ** -11)]])
    bmax = (targets.astype(np.float64) * 6.0).astype(np.float32)
    nb = bmax.size
    blocks = np.zeros((((nb + 4) // 4) * 4, 16), np.float32)
    blocks[:nb, 0] = bmax
    blocks[:nb, 1:] = bmax[:, None] * np.linspace(-1, 1, 15, dtype=np.float32)[None, :]
    blocks[nb, 0] = 2688.0                           # gsa = 1
    x = blocks.reshape(-1, 64)
    _check_exact(x, to_device(x, "f32"))


@pytest.mark.parametrize("scale", [0.0, 1e-30, 1e-20, 1.0, 1e20, 1e30])
def test_magnitude_edges_fp32(scale):
    """gsa == 0, gsa below / above the division shortcut's range, subnormal inputs."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((5, 128)) * scale).astype(np.float32)
    x[1, :16] = 0.0
    x[2, 3] = np.float32(1e-40) if scale else 0.0    # a subnormal element
    x[3, 17] = -np.float32(1e-42) if scale else 0.0
    _check_exact(x, to_device(x, "f32"))


def test_bf16_subnormals_and_signed_zero():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    bits = WL.float32_to_bf16_bits(x)
    bits[0, :8] = np.arange(1, 9, dtype=np.uint16)           # positive bf16 subnormals
    bits[1, :8] = np.arange(1, 9, dtype=np.uint16) | 0x8000  # negative subnormals
    bits[2, :4] = 0x8000                                     # -0.0
    _check_exact(WL.bf16_bits_to_float32(bits), to_device(bits, "bf16"))
    tiny = bits.copy()
    tiny[:] = np.arange(tiny.size, dtype=np.uint16).reshape(tiny.shape) % 64  # only subnormals
    _check_exact(WL.bf16_bits_to_float32(tiny), to_device(tiny, "bf16"))


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_pack_weight(name):
    import nvfp4_router_gate_gb300 as R
    w = WL.WORKLOADS[name]
    W = WL.make_w(w)
    c, s, g = R.nvfp4_pack_weight(to_device(W, w.dtype))
    torch.cuda.synchronize()
    q, sb, gg = Q.quantize(as_f32(W, w.dtype))
    assert f32_bits(g.cpu().numpy()[0]) == f32_bits(gg)
    assert np.array_equal(c.cpu().numpy(), Q.pack_fp4(q))
    assert np.array_equal(s.cpu().numpy(), Q.sf_to_tiles(sb))


def test_repeated_calls_same_workspace():
    """Tickets return to zero: many calls of different sizes on one workspace."""
    import nvfp4_router_gate_gb300 as R
    ws = R.new_workspace(R.nvfp4_quantize_workspace_size(4096, 7168))
    for seed, T in enumerate([4096, 3, 700, 1, 4096]):
        rng = np.random.default_rng(seed)
        x = rng.standard_normal((T, 7168)).astype(np.float32) * (seed + 1)
        c, s, g = R.nvfp4_quantize_act(to_device(x, "f32"), workspace=ws)
        torch.cuda.synchronize()
        q, sb, gg = Q.quantize(x)
        assert f32_bits(g.cpu().numpy()[0]) == f32_bits(gg)
        assert np.array_equal(c.cpu().numpy(), Q.pack_fp4(q))
    assert R.nvr_read_device_status(ws) == 0
