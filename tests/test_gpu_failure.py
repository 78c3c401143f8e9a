"""Failure detection on the GPU without a fault: a bounded device wait that
nothing satisfies gives up, the error word reports GDN_ERR_DEVICE_TIMEOUT, and
the context keeps working (gdn_selftest_wait_timeout in include/gdn.h)."""
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_step, gdn_selftest_wait_timeout,
                                                    gdn_stream_status, inputs)

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_stays_usable():
    assert gdn_stream_status() == "GDN_OK"
    gdn_selftest_wait_timeout(2000)          # 2 ms, then the kernel returns
    assert gdn_stream_status() == "GDN_ERR_DEVICE_TIMEOUT"
    assert gdn_stream_status() == "GDN_OK"   # read and cleared
    # the next launches run normally
    d = inputs.make_decode(4, 2, 4, 64, 64, "bf16", seed=7)
    x = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    o = gdn_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"])
    assert gdn_stream_status() == "GDN_OK"
    assert torch.isfinite(o.float()).all()


def test_selftest_on_a_side_stream():
    s = torch.cuda.Stream()
    gdn_selftest_wait_timeout(500, stream=s)
    assert gdn_stream_status(s) == "GDN_ERR_DEVICE_TIMEOUT"
    assert gdn_stream_status(s) == "GDN_OK"
