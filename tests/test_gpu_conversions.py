"""Exhaustive check of the two hardware conversions behind every quantizer
path -- float32 -> E2M1 codes and float32 -> E4M3 scale bytes, round to
nearest even, saturating -- on every float32 bit pattern but the NaNs.  The
expected code of each input comes from the oracle's encoders as step
functions (their rounding thresholds, `oracle.formats.e2m1_thresholds` /
`e4m3_thresholds`, pinned on the CPU to the ties-to-even midpoints of the
printed format tables); the GPU kernel only converts and compares."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

from oracle import formats  # noqa: E402


def test_every_float32_converts_as_the_oracle_encodes():
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    th2 = torch.from_numpy(formats.e2m1_thresholds().view(np.int32)).cuda()
    th8 = torch.from_numpy(formats.e4m3_thresholds().view(np.int32)).cuda()
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    first = torch.zeros(2, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    _native.check("nvr_test_conversion_sweep",
                  lib.nvr_test_conversion_sweep(th2.data_ptr(), th8.data_ptr(), counts.data_ptr(),
                                                first.data_ptr(), stream))
    torch.cuda.synchronize()
    bad2, bad8, checked = (int(v) for v in counts.cpu())
    f2, f8 = (int(v) & 0xFFFFFFFF for v in first.cpu())
    assert checked == 2 ** 32 - 2 * (2 ** 23 - 1)        # every pattern but the 2^24 - 2 NaNs
    assert bad2 == 0, "E2M1: %d mismatches, first at bits 0x%08x" % (bad2, f2)
    assert bad8 == 0, "E4M3: %d mismatches, first at bits 0x%08x" % (bad8, f8)
    assert f2 == 0xFFFFFFFF and f8 == 0xFFFFFFFF


def test_sweep_reports_a_planted_threshold_error():
    """A threshold moved by one float32 (an oracle mistake planted on the CPU
    side of the comparison) shows up as exactly the inputs it misclassifies:
    the +/- pair at the old threshold."""
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    t2 = formats.e2m1_thresholds().copy()
    t2[3] += 1                                            # the tie at 1.75 sent the wrong way
    th2 = torch.from_numpy(t2.view(np.int32)).cuda()
    th8 = torch.from_numpy(formats.e4m3_thresholds().view(np.int32)).cuda()
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    first = torch.zeros(2, dtype=torch.int32, device="cuda")
    _native.check("nvr_test_conversion_sweep",
                  lib.nvr_test_conversion_sweep(th2.data_ptr(), th8.data_ptr(), counts.data_ptr(),
                                                first.data_ptr(), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    bad2, bad8, _ = (int(v) for v in counts.cpu())
    assert bad2 == 2 and bad8 == 0
    assert int(first[0].item()) & 0xFFFFFFFF == int(formats.e2m1_thresholds()[3])
