"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/gdn.h declares, and rejects host-checkable errors without launching
anything (these calls touch no GPU)."""
import ctypes
import os
import re

import pytest

from gated_deltanet_linear_recurrence_gb300 import _lib
from gated_deltanet_linear_recurrence_gb300.build import build, ROOT

HEADER = os.path.join(ROOT, "include", "gdn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "gdn_prefill" in names and "gdn_decode_step" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in gdn.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.gdn_status_string(code).decode() == name


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=None, state_out=FAKE, o=FAKE,
             cu=FAKE, n=1, t=64, h_k=1, h_v=1, d_k=16, d_v=16, dtype=1, scale=1.0, algo=1,
             ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.gdn_prefill(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state_in"],
                           a["state_out"], a["o"], a["cu"], a["n"], a["t"], a["h_k"], a["h_v"],
                           a["d_k"], a["d_v"], a["dtype"], a["scale"], a["algo"], a["ws"],
                           a["ws_bytes"], a["stream"])


def test_options_host_errors(lib):
    """Unknown option bits are refused before anything is launched."""
    assert lib.gdn_prefill_ex(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 64, 1, 1,
                              16, 16, 1, 1.0, 1, None, 0, 4, None) == 2
    assert lib.gdn_prefill_ex(None, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 64, 1, 1,
                              16, 16, 1, 1.0, 1, None, 0, 1, None) == 1
    assert lib.gdn_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 16, 16, 1,
                                  1.0, 8, None) == 2
    assert lib.gdn_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 1, 1, 16, 16, 1,
                                  1.0, 1, None) == 1


def test_prefill_host_errors(lib):
    assert prefill(lib, q=None) == 1                     # NULL
    assert prefill(lib, cu=None) == 1
    assert prefill(lib, n=-1) == 2                       # negative
    assert prefill(lib, algo=7) == 2                     # bad enum
    assert prefill(lib, dtype=5) == 4
    assert prefill(lib, d_k=48) == 3                     # head dim not supported
    assert prefill(lib, h_k=2, h_v=3) == 3               # h_v % h_k
    assert prefill(lib, t=1 << 31) == 3                  # beyond int32 cu_seqlens
    assert prefill(lib, k=FAKE + 4) == 5                 # misaligned
    assert prefill(lib, state_in=FAKE + 16, state_out=FAKE) == 2   # partial overlap
    assert prefill(lib, n=0) == 0                        # nothing to do: OK, no launch
    assert prefill(lib, n=0, q=None) == 0
    chunk = dict(d_k=128, d_v=32)                        # a shape the chunked kernels cover
    assert prefill(lib, algo=4, **chunk) == 1            # two-kernel form without workspace
    assert prefill(lib, algo=4, ws=FAKE, ws_bytes=16, **chunk) == 7
    assert prefill(lib, algo=4, ws=FAKE + 8, ws_bytes=1 << 30, **chunk) == 5
    assert prefill(lib, algo=3, dtype=0, **chunk) == 4   # chunked forms are bf16 only
    assert prefill(lib, algo=3, d_k=64, d_v=32) == 3     # the fused kernel needs d_k = 128
    assert prefill(lib, algo=4, d_k=32, d_v=32, ws=FAKE, ws_bytes=1 << 30) == 3  # d_k 64 or 128


def test_noalloc_host_errors(lib):
    """The allocation-free prefill refuses, without touching a device, problems
    whose scratch exceeds its fixed array and arguments gdn_prefill refuses."""
    def call(n=1, t=64, h_k=1, h_v=2, d_k=128, d_v=32, dtype=1):
        return lib.gdn_prefill_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, n, t,
                                       h_k, h_v, d_k, d_v, dtype, 1.0, None)
    big = 1 << 20   # 1M tokens at 2 value heads: ~1.1 GB of scratch
    assert lib.gdn_prefill_workspace_size(1, big, 1, 2, 128, 32, 1, 4) > 128 << 20
    assert lib.gdn_prefill_workspace_size(1, 4096, 16, 32, 128, 128, 1, 4) <= 128 << 20
    assert call(t=big) == 7                              # GDN_ERR_WORKSPACE_TOO_SMALL
    assert call(d_k=32) == 3                             # chunked needs d_k 64 or 128
    assert call(dtype=0) == 4                            # and bf16
    assert call(n=-1) == 2


def decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, o=FAKE, b=1, h_k=1, h_v=1,
             d_k=16, d_v=16, dtype=1, scale=1.0, stream=None)
    a.update(kw)
    return lib.gdn_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state"], a["o"],
                               a["b"], a["h_k"], a["h_v"], a["d_k"], a["d_v"], a["dtype"],
                               a["scale"], a["stream"])


def test_decode_host_errors(lib):
    assert decode(lib, state=None) == 1
    assert decode(lib, b=-2) == 2
    assert decode(lib, d_v=8) == 3
    assert decode(lib, h_k=4, h_v=2) == 3
    assert decode(lib, dtype=3) == 4
    assert decode(lib, o=FAKE + 2) == 5
    assert decode(lib, b=0) == 0


def test_workspace_and_crossover_queries(lib):
    assert lib.gdn_prefill_workspace_size(1, 4096, 16, 32, 128, 128, 1, 1) == 0  # scan needs none
    ws = lambda n, t, algo: lib.gdn_prefill_workspace_size(n, t, 16, 32, 128, 128, 1, algo)
    assert ws(1, 4096, 3) == 0                           # fused chunked kernel: none
    # long sequences: two kernels, or the cooperative form (the same plus its flags)
    assert ws(1, 4096, 2) == ws(1, 4096, 5) > ws(1, 4096, 4) > 0
    assert ws(1, 200, 2) == 0 and ws(1, 200, 0) == 0     # one 200-token prompt: fused
    assert ws(1, 200, 4) > 0                             # unless the two kernels are forced
    # four prompts at 32 value heads: the table takes the two kernels from any length
    assert ws(4, 1000, 0) == ws(4, 1000, 5) > 0
    assert ws(4, 2048, 2) == ws(4, 2048, 5) > ws(4, 2048, 4) > 0
    # header (1 KB-rounded) + I = (T/64 + N + 1) x h_v per-chunk packages of 57 KB
    items = (2048 // 64 + 5) * 32
    assert ws(4, 2048, 4) == 1024 + items * 58368
    # the cooperative form adds one ready flag per item and a counter, 1 KB-rounded
    assert ws(4, 2048, 5) == ws(4, 2048, 4) + ((items + 1) * 4 + 1023) // 1024 * 1024
    x = lib.gdn_prefill_crossover_tokens(16, 32, 128, 128, 1)
    assert x > 0
    assert lib.gdn_prefill_crossover_tokens(16, 32, 128, 48, 1) == 2**31 - 1


def test_streamed_host_errors(lib):
    """gdn_prefill_streamed refuses bad arguments before launching anything."""
    def call(t=4096, piece=1024, h_k=16, h_v=32, d_k=128, d_v=128, dtype=1, ws=FAKE,
             ws_bytes=1 << 40, opts=0, **ptr):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=None, state_out=FAKE, o=FAKE)
        p.update(ptr)
        return lib.gdn_prefill_streamed(p["q"], p["k"], p["v"], p["g"], p["beta"], p["state_in"],
                                        p["state_out"], p["o"], t, h_k, h_v, d_k, d_v, dtype, 1.0,
                                        piece, ws, ws_bytes, opts, None)
    assert call(piece=1000) == 2                         # not whole chunks
    assert call(opts=6, ws_bytes=4096) in (2, 7)          # an unknown option bit or the size
    assert call(piece=0) == 2
    assert call(t=-1) == 2
    assert call(d_k=48) == 3
    assert call(h_k=3, h_v=4) == 3
    assert call(q=None) == 1
    assert call(ws=None) == 1
    assert call(ws=FAKE + 8) == 5
    assert call(k=FAKE + 4) == 5
    assert call(ws_bytes=4096) == 7                      # GDN_ERR_WORKSPACE_TOO_SMALL
    assert call(state_in=FAKE + 64) == 2                 # partial overlap with state_out
    size = lib.gdn_prefill_streamed_workspace_size
    assert size(1000, 16, 32, 128, 128, 1) == 0
    # bounded by the piece: the same for any prompt length, and far below the whole
    # prompt's workspace for a 128K-token prompt
    assert size(8192, 16, 32, 128, 128, 1) == 256 + lib.gdn_prefill_workspace_size(
        1, 8192, 16, 32, 128, 128, 1, 4)
    assert size(8192, 16, 32, 128, 128, 1) * 10 < lib.gdn_prefill_workspace_size(
        1, 131072, 16, 32, 128, 128, 1, 4)


def test_decode_multi_host_errors(lib):
    def call(b=2, n=3, h_k=1, h_v=1, d_k=16, d_v=16, dtype=1, snap=None, opts=0, **ptr):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, o=FAKE)
        p.update(ptr)
        return lib.gdn_decode_multi(p["q"], p["k"], p["v"], p["g"], p["beta"], p["state"], p["o"],
                                    snap, b, n, h_k, h_v, d_k, d_v, dtype, 1.0, opts, None)
    assert call(n=0) == 2
    assert call(n=2000) == 2
    assert call(b=-1) == 2
    assert call(d_k=8) == 3
    assert call(dtype=4) == 4
    assert call(state=None) == 1
    assert call(o=FAKE + 2) == 5
    assert call(snap=FAKE + 16) == 2                     # snapshots overlap the state
    assert call(opts=2) == 2                             # unknown option bit
    assert call(b=0) == 0


def attn(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, lens=FAKE, o=FAKE, b=1, h_q=16, h_kv=2, d=256, cap=4096,
             dtype=1, scale=0.0625, layout=0, bk=0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.gdn_attn_decode(a["q"], a["k"], a["v"], a["lens"], a["o"], a["b"], a["h_q"],
                               a["h_kv"], a["d"], a["cap"], a["dtype"], a["scale"], a["layout"],
                               a["bk"], a["ws"], a["ws_bytes"], a["stream"])


def test_attn_decode_host_errors(lib):
    """Decode attention: every host-checkable error returns before any device call."""
    assert attn(lib, q=None) == 1
    assert attn(lib, lens=None) == 1
    assert attn(lib, k=None) == 1                         # cache pointers needed when capacity > 0
    assert attn(lib, b=-1) == 2
    assert attn(lib, cap=-1) == 2
    assert attn(lib, layout=3) == 2                       # bad enum
    assert attn(lib, bk=100) == 2                         # not a multiple of 64
    assert attn(lib, bk=-64) == 2
    assert attn(lib, d=128) == 3                          # head dim 256 only
    assert attn(lib, h_q=16, h_kv=3) == 3                 # h_q % h_kv
    assert attn(lib, h_q=32, h_kv=2) == 3                 # more than 8 query heads per KV head
    assert attn(lib, b=1024, h_kv=2, h_q=16, cap=1 << 21) == 3   # cache rows beyond int32
    assert attn(lib, dtype=0) == 4                        # bf16 only
    assert attn(lib, o=FAKE + 8) == 5
    assert attn(lib, lens=FAKE + 2) == 5
    assert attn(lib, b=0) == 0                            # nothing to do
    assert attn(lib, b=0, q=None) == 0


def test_attn_workspace_size(lib):
    """Workspace bound: 0 for the general layout, else B x h_q x n x (D + 2) x 4
    with n = ceil(capacity / block), block 128 when the library picks it."""
    f = lib.gdn_attn_decode_workspace_size
    assert f(1, 16, 2, 256, 131072, 1, 0) == 0
    assert f(1, 16, 2, 256, 131072, 2, 2048) == 1 * 16 * 64 * 258 * 4
    assert f(3, 16, 2, 256, 131072, 0, 0) == 3 * 16 * 1024 * 258 * 4
    assert f(2, 8, 1, 256, 1000, 2, 512) == 2 * 8 * 2 * 258 * 4
    assert f(2, 8, 1, 256, 512, 2, 512) == 0              # a single block needs no merge
    assert f(1, 16, 2, 128, 4096, 0, 0) == 0              # invalid shape
    assert f(1, 16, 2, 256, 4096, 2, 100) == 0            # invalid block


def test_prefill_from_host_memory_errors(lib):
    """gdn_prefill_host: host-checkable errors return before any device call."""
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, si=None, so=FAKE, o=FAKE, t=4096,
                 h_k=16, h_v=32, d_k=128, d_v=128, dtype=1, scale=1.0, piece=1024, ws=FAKE,
                 ws_bytes=1 << 40, opt=0, stream=None)
        a.update(kw)
        return lib.gdn_prefill_host(a["q"], a["k"], a["v"], a["g"], a["beta"], a["si"], a["so"],
                                    a["o"], a["t"], a["h_k"], a["h_v"], a["d_k"], a["d_v"],
                                    a["dtype"], a["scale"], a["piece"], a["ws"], a["ws_bytes"],
                                    a["opt"], a["stream"])
    assert call(piece=100) == 2                          # not a multiple of 64
    assert call(piece=0) == 2
    assert call(t=-1) == 2
    assert call(opt=4) == 2                              # unknown option bit
    assert call(dtype=7) == 4
    assert call(d_k=48) == 3
    assert call(h_k=3, h_v=32) == 3
    assert call(q=None) == 1
    assert call(so=None) == 1
    assert call(ws=None) == 1
    assert call(ws=FAKE + 8) == 5
    assert call(ws_bytes=1024) == 7                      # workspace too small
    need = lib.gdn_prefill_host_workspace_size(1024, 16, 32, 128, 128, 1)
    assert need > 0 and call(ws_bytes=need - 1) == 7
    assert lib.gdn_prefill_host_workspace_size(100, 16, 32, 128, 128, 1) == 0
    # grows with the piece, not with the prompt
    assert lib.gdn_prefill_host_workspace_size(2048, 16, 32, 128, 128, 1) > need


def test_prefill_form_query(lib):
    """gdn_prefill_form reports the evaluation a call would run, from sizes alone
    (the SM count given, so no device is needed)."""
    S = 152  # SMs of a GB300

    def form(n, t, algo=0, ws=None, opt=0, sms=S, d_v=128, dtype=1):
        if ws is None:
            ws = lib.gdn_prefill_workspace_size(n, t, 16, 32, 128, d_v, dtype, algo)
        return lib.gdn_prefill_form(n, t, 16, 32, 128, d_v, dtype, algo, ws, opt, sms)

    SCAN, FUSED, SPLIT, COOP = 1, 3, 4, 5
    x = lib.gdn_prefill_crossover_tokens(16, 32, 128, 128, 1)
    assert form(1, x - 1) == SCAN                       # below the crossover: token scan
    assert form(1, 200) == FUSED                        # short: the fused kernel, no workspace
    assert form(1, 2048) == SPLIT                       # two kernels
    assert form(1, 4096) == COOP                        # from 4,096 tokens: cooperative
    assert form(1, 4096, ws=0) == FUSED                 # no workspace: the fused kernel
    split_ws = lib.gdn_prefill_workspace_size(1, 4096, 16, 32, 128, 128, 1, 4)
    assert form(1, 4096, ws=split_ws) == SPLIT          # no room for the ready flags
    assert form(1, 4096, sms=64) == SPLIT               # 64 state passes need > 96 SMs
    # state passes of 64 rows: 2 x 32 x 2 = 128 are more than two thirds of the SMs
    assert form(2, 2 * 4096) == SPLIT
    # few value heads: the table (measured at 4 value heads) never takes the
    # cooperative form, whose 64-row state passes lose to the two kernels' 32-row ones
    ws8 = lib.gdn_prefill_workspace_size(4, 4 * 4096, 4, 8, 128, 128, 1, 0)
    assert lib.gdn_prefill_form(4, 4 * 4096, 4, 8, 128, 128, 1, 0, ws8, 0, S) == SPLIT
    assert lib.gdn_prefill_form(4, 4 * 4096, 4, 8, 128, 128, 1, 5, ws8, 0, S) == COOP  # forced
    assert form(1, 4096, algo=4) == SPLIT               # forced forms
    assert form(1, 2048, algo=5) == COOP
    assert form(1, 4096, algo=3) == FUSED
    assert form(1, 4096, algo=1) == SCAN
    assert form(1, 4096, opt=1, ws=0) == SCAN           # normalisation without room: scan
    assert form(1, 4096, d_v=16, ws=1 << 30) == SCAN    # d_v below the chunked kernels' 32
    assert form(0, 0) == SCAN                           # nothing runs
    # refusals come back negated
    assert form(1, 4096, algo=5, ws=0) == -1            # the cooperative form needs a workspace
    assert form(1, 4096, algo=5, ws=1024) == -7
    assert form(1, 4096, algo=4, ws=0) == -1
    assert form(1, 4096, algo=3, opt=1) == -2           # fused kernel has no normalisation
    assert form(1, 4096, algo=2, dtype=0) == -4         # fp32 has no chunked evaluation
    assert form(1, 4096, algo=9) == -2
    assert form(-1, 4096) == -2
    assert lib.gdn_prefill_form(1, 4096, 16, 30, 128, 128, 1, 0, 0, 0, S) == -3
    # d_k = 64: the two-kernel and cooperative forms (Q and K zero-padded to 128
    # columns); no fused kernel, so without a workspace AUTO scans
    def form64(n, t, algo=0, ws=None, d_k=64):
        if ws is None:
            ws = lib.gdn_prefill_workspace_size(n, t, 16, 32, d_k, 128, 1, algo)
        return lib.gdn_prefill_form(n, t, 16, 32, d_k, 128, 1, algo, ws, 0, S)
    assert lib.gdn_prefill_workspace_size(1, 200, 16, 32, 64, 128, 1, 0) > 0
    assert form64(1, 200) == SPLIT
    assert form64(1, 8192) == COOP
    assert form64(1, 200, ws=0) == SCAN
    assert form64(1, 200, algo=2, ws=0) == -7           # CHUNKED without room for two kernels
    assert form64(1, 200, algo=3) == -3                 # no fused kernel for d_k = 64
    assert form64(1, 200, d_k=32) == SCAN               # d_k 32: the token scan
    assert form64(1, 200, algo=2, d_k=32) == -3


def test_prefill_form_python_names():
    """The Python wrapper maps the query's answer to the algorithm names that
    gdn_prefill takes, and raises GdnError for refused arguments."""
    import torch
    from gated_deltanet_linear_recurrence_gb300 import (GdnError, gdn_prefill_form,
                                                        gdn_prefill_workspace_size)

    ws = gdn_prefill_workspace_size(1, 4096, 16, 32, 128, 128, torch.bfloat16)
    f = lambda t, **kw: gdn_prefill_form(1, t, 16, 32, 128, 128, torch.bfloat16, sm_count=152, **kw)
    assert f(4096, workspace_bytes=ws) == "chunked_coop"
    assert f(2048, workspace_bytes=ws) == "chunked_split"
    assert f(4096) == "chunked_fused"
    assert f(4, workspace_bytes=ws) == "scan"
    assert f(4096, algo="chunked_split", workspace_bytes=ws) == "chunked_split"
    with pytest.raises(GdnError):
        f(4096, algo="chunked_coop")          # no workspace
    with pytest.raises(GdnError):
        f(4096, algo="chunked_fused", qk_l2norm=True)


def test_output_norm_host_errors(lib):
    """The output RMS normalisation entry points refuse bad arguments before
    launching anything (no device is touched)."""
    def dec(b=2, h_k=1, h_v=2, d_k=16, d_v=16, dtype=1, eps=1e-6, w=None, opts=0, **ptr):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, o=FAKE)
        p.update(ptr)
        return lib.gdn_decode_step_rmsnorm(p["q"], p["k"], p["v"], p["g"], p["beta"], p["state"],
                                           p["o"], w, eps, b, h_k, h_v, d_k, d_v, dtype, 1.0,
                                           opts, None)
    assert dec(b=0) == 0                      # nothing to do
    assert dec(b=-1) == 2
    assert dec(eps=-1.0) == 2                 # eps must be >= 0
    assert dec(eps=float("nan")) == 2
    assert dec(opts=4) == 2
    assert dec(dtype=7) == 4
    assert dec(d_v=48) == 3
    assert dec(o=None) == 1
    assert dec(w=FAKE + 4) == 5               # misaligned weight

    def norm(rows=4, h_v=2, d_v=64, dtype=1, eps=1e-6, o=FAKE, w=None):
        return lib.gdn_output_rmsnorm(o, w, rows, h_v, d_v, dtype, eps, None)
    assert norm(rows=0) == 0
    assert norm(rows=-1) == 2
    assert norm(h_v=0) == 2
    assert norm(eps=-0.5) == 2
    assert norm(d_v=24) == 3
    assert norm(dtype=3) == 4
    assert norm(o=None) == 1
    assert norm(o=FAKE + 2) == 5
    assert norm(w=FAKE + 8) == 5
