"""gdn_prefill_noalloc, the entry point that allocates nothing (its scratch is
a fixed array the library holds in device memory), against gdn_prefill with a
caller workspace: two calls in a row through the C ABI.  This file runs last
and passes alone in a fresh process too."""
import ctypes

import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (NOALLOC_SCRATCH_BYTES, _lib, gdn_prefill,
                                                    gdn_prefill_workspace_size,
                                                    gdn_stream_status, inputs)
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu

TIGHT = 8e-3  # the chunked tests' tolerance


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def call_noalloc(lib, x, o, st, scale):
    T, h_k, d_k = x["q"].shape
    h_v, d_v = x["v"].shape[1], x["v"].shape[2]
    N = x["cu_seqlens"].numel() - 1
    sin = x["state_in"]
    return lib.gdn_prefill_noalloc(
        x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["g"].data_ptr(),
        x["beta"].data_ptr(), None if sin is None else sin.data_ptr(), st.data_ptr(),
        o.data_ptr(), x["cu_seqlens"].data_ptr(), N, T, h_k, h_v, d_k, d_v, _lib.GDN_BF16,
        ctypes.c_float(scale), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_gdn_prefill_two_calls_in_a_row():
    lib = _lib.load()
    cases = [  # the larger first, so the second call runs over the first call's leftovers
        (inputs.make_prefill([4096], 16, 32, 128, 128, "bf16", seed=31), 1.0),
        (inputs.make_prefill([300, 1, 777, 0, 64], 2, 4, 128, 64, "bf16", seed=32,
                             state_std=0.05), 0.7),
    ]
    for d, scale in cases:
        x = dev(d)
        T, N = x["q"].shape[0], x["cu_seqlens"].numel() - 1
        h_k, h_v, d_v = x["q"].shape[1], x["v"].shape[1], x["v"].shape[2]
        assert gdn_prefill_workspace_size(N, T, h_k, h_v, 128, d_v,
                                          algo="chunked_split") <= NOALLOC_SCRATCH_BYTES
        o_ref, st_ref = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                                    state_in=x["state_in"], scale=scale, algo="chunked_split")
        o = torch.full_like(o_ref, float("nan"))
        st = torch.full_like(st_ref, float("nan"))
        assert call_noalloc(lib, x, o, st, scale) == _lib.GDN_OK
        assert gdn_stream_status() == "GDN_OK"
        eo = rel_l2(to_np(o), to_np(o_ref))
        es = rel_l2(to_np(st), to_np(st_ref))
        assert eo < TIGHT and es < TIGHT, (eo, es)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    x = dev(inputs.make_prefill([64], 1, 2, 128, 32, "bf16", seed=33))
    o = torch.empty((64, 2, 32), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((1, 2, 32, 128), dtype=torch.float32, device="cuda")
    T_big = 1 << 20  # 1M tokens at 2 value heads: ~1.1 GB of scratch
    assert gdn_prefill_workspace_size(1, T_big, 1, 2, 128, 32,
                                      algo="chunked_split") > NOALLOC_SCRATCH_BYTES
    rc = lib.gdn_prefill_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                 x["g"].data_ptr(), x["beta"].data_ptr(), None, st.data_ptr(),
                                 o.data_ptr(), x["cu_seqlens"].data_ptr(), 1, T_big, 1, 2, 128,
                                 32, _lib.GDN_BF16, ctypes.c_float(1.0), None)
    assert _lib.STATUS_NAMES[rc] == "GDN_ERR_WORKSPACE_TOO_SMALL"
    assert gdn_stream_status() == "GDN_OK"
