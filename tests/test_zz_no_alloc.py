"""gdn_prefill_noalloc, the entry point that allocates nothing (its scratch is
a fixed array the library holds in device memory), against gdn_prefill with a
caller workspace, through the C ABI.

Both run the same deterministic two-kernel chunked evaluation on the same
inputs, so their outputs must agree bit for bit; a mistake in handing the
fixed array over as the workspace would show as a difference.  The calls run
back to back on one stream with no synchronisation between them (two
one-sequence calls, then a many-sequence one), so each call runs over the
previous call's leftovers in the shared array, and the device's free memory
and the torch allocator's counters are checked to be unchanged across them.
This file runs last and passes alone in a fresh process too."""
import ctypes

import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (NOALLOC_SCRATCH_BYTES, _lib, gdn_prefill,
                                                    gdn_prefill_workspace_size,
                                                    gdn_stream_status, inputs)

pytestmark = pytest.mark.gpu


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


def allocator_counters():
    s = torch.cuda.memory_stats()
    return (s.get("allocation.all.allocated", 0), s.get("segment.all.allocated", 0),
            s.get("reserved_bytes.all.current", 0))


def test_noalloc_matches_gdn_prefill_bitwise_back_to_back():
    lib = _lib.load()
    cases = [  # the largest first, so the later calls run over its leftovers
        (inputs.make_prefill([4096], 16, 32, 128, 128, "bf16", seed=31), 1.0),
        (inputs.make_prefill([1000], 2, 4, 128, 64, "bf16", seed=34, state_std=0.05), 0.9),
        (inputs.make_prefill([300, 1, 777, 0, 64], 2, 4, 128, 64, "bf16", seed=32,
                             state_std=0.05), 0.7),
    ]
    runs = []
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
        runs.append((x, scale, o, st, o_ref, st_ref))
    # one call first: the per-device set-up (the array's address) happens there
    x, scale, o, st = runs[-1][:4]
    assert call_noalloc(lib, x, o, st, scale) == _lib.GDN_OK
    assert gdn_stream_status() == "GDN_OK"
    for r in runs:
        r[2].fill_(float("nan"))
        r[3].fill_(float("nan"))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    counters0 = allocator_counters()
    for x, scale, o, st, _, _ in runs:  # back to back on one stream
        assert call_noalloc(lib, x, o, st, scale) == _lib.GDN_OK
    assert gdn_stream_status() == "GDN_OK"
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "device memory changed across the calls"
    assert allocator_counters() == counters0, "the torch allocator was used"
    for x, scale, o, st, o_ref, st_ref in runs:
        assert torch.equal(o, o_ref)
        assert torch.equal(st, st_ref)


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
