"""The measured crossover table (AUTO's choice of evaluation by shape): for four
shapes whose fastest form differs, AUTO runs the form the table names, that
form is the fastest of all forms timed live on this GPU (within timing noise),
and AUTO's output matches the fp64 oracle."""
import statistics

import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill, gdn_prefill_form,
                                                    gdn_prefill_workspace_size,
                                                    gdn_stream_status, inputs)
from tests.test_gpu_chunked import TIGHT, dev, full_errors

pytestmark = pytest.mark.gpu

# (lengths, h_k, h_v, d_k, d_v, the form the table picks)
CASES = [
    ([4096], 16, 32, 128, 128, "chunked_coop"),       # one long prompt, many heads
    ([2048], 2, 4, 128, 128, "chunked_split"),        # few heads: 32-row state passes win
    ([128] * 4, 16, 32, 128, 32, "chunked_fused"),    # short prompts: one kernel, no workspace
    ([16] * 16, 16, 32, 64, 32, "scan"),              # very short, d_k = 64: the token scan
]


def timed(fn, reps=7):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    buf = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    ts = []
    for i in range(reps + 2):
        buf.fill_(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        if i >= 2:
            ts.append(a.elapsed_time(b))
    return statistics.median(ts)


@pytest.mark.parametrize("lengths,h_k,h_v,d_k,d_v,want", CASES)
def test_auto_runs_the_fastest_form(lengths, h_k, h_v, d_k, d_v, want):
    d = inputs.make_prefill(lengths, h_k, h_v, d_k, d_v, "bf16", seed=len(lengths) + d_v + d_k)
    x = dev(d)
    N, T = len(lengths), sum(lengths)
    ws_auto = gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v, torch.bfloat16, "auto")
    assert gdn_prefill_form(N, T, h_k, h_v, d_k, d_v, torch.bfloat16, "auto", ws_auto) == want
    ws = torch.empty(max(gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v, torch.bfloat16,
                                                    "chunked_coop"), 16),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((N, h_v, d_v, d_k), dtype=torch.float32, device="cuda")
    forms = ["scan", "chunked_split"]
    if d_k == 128:
        forms.append("chunked_fused")
    if want == "chunked_coop":
        forms.append("chunked_coop")
    times = {}
    for f in forms:
        times[f] = timed(lambda: gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                             x["cu_seqlens"], state_out=st, o=o, algo=f,
                                             workspace=ws))
        assert gdn_stream_status() == "GDN_OK"
    best = min(times.values())
    assert times[want] <= 1.1 * best + 2e-3, times  # ms; event timing noise
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], state_out=st, o=o,
                algo="auto", workspace=ws[:ws_auto] if ws_auto else None)
    assert gdn_stream_status() == "GDN_OK"
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)
