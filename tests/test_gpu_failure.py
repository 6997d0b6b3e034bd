"""Device-side failure detection without a GPU fault.

Every wait in the tensor-core kernel is bounded (about one second).  The test
hook oop_debug_inject_timeout makes the next launch skip one of its TMA
copies, so its MMA thread waits for data that never comes: the kernel must
give up, record OOP_ERR_DEVICE_TIMEOUT in the device status word, release its
tensor memory and return -- and the context must stay usable.
"""

import time

import numpy as np
import pytest

import synth
from helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


@pytest.mark.parametrize("tid", [synth.TYPE_Q8_0, synth.TYPE_F32])
def test_bounded_wait_reports_timeout(op, orc, tid):
    import torch
    ne_a, ne_b = (256, 128, 1, 1), (128, 128, 1, 1)
    a = synth.make_a(tid, ne_a, 70, std=0.02)
    b = synth.make_b(ne_b, 71, std=1e3, outliers=True)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    assert op.device_status(clear=True) == op.OK
    assert op.lib().oop_debug_inject_timeout(1) == op.OK
    t0 = time.time()
    op.out_prod(ta, tb, a_type=tid, ne_a=ne_a, path=op.PATH_TCGEN05)
    st = op.device_status(clear=True)
    elapsed = time.time() - t0
    assert st == op.ERR_DEVICE_TIMEOUT, op.status_string(st)
    assert elapsed < 30.0
    assert op.device_status() == op.OK            # cleared
    # the hook is consumed by one launch; the next call is normal and correct
    ref = orc.out_prod(a, tid, b, ne_a, ne_b)
    out = op.out_prod(ta, tb, a_type=tid, ne_a=ne_a, path=op.PATH_TCGEN05)
    torch.cuda.synchronize()
    assert op.device_status() == op.OK
    assert_parity(out.cpu().numpy(), ref["f64"], ref["abs"], "after timeout")
