"""GB300-native (sm_103a) Gated DeltaNet recurrence.

Python face of the C ABI in include/gdn.h.  The functions below carry the
ABI's names; they take torch CUDA tensors (PyTorch supplies device memory and
streams), marshal pointers and sizes, and call the CUDA library.  Outputs not
passed in are allocated with torch.  Nothing here computes the recurrence.

    S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t (scale q_t)
"""
import torch

from . import _lib
from ._lib import GdnError, STATUS_NAMES

__all__ = ["gdn_prefill", "gdn_prefill_streamed", "gdn_prefill_streamed_workspace_size",
           "gdn_prefill_host", "gdn_prefill_host_workspace_size",
           "gdn_prefill_noalloc", "gdn_decode_step", "gdn_decode_step_rmsnorm",
           "gdn_output_rmsnorm", "gdn_decode_multi", "gdn_attn_decode",
           "gdn_attn_decode_workspace_size", "gdn_attn_decode_block_keys",
           "gdn_prefill_workspace_size",
           "gdn_stream_status", "gdn_status_string", "gdn_prefill_crossover_tokens",
           "gdn_prefill_form", "gdn_selftest_wait_timeout", "GdnError",
           "STATUS_NAMES", "NOALLOC_SCRATCH_BYTES"]

NOALLOC_SCRATCH_BYTES = 128 << 20  # GDN_NOALLOC_SCRATCH_BYTES in include/gdn.h

_DTYPES = {torch.float32: _lib.GDN_F32, torch.bfloat16: _lib.GDN_BF16}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t):
    if t.dtype not in _DTYPES:
        raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")
    return _DTYPES[t.dtype]


def _require(cond, msg):
    if not cond:
        raise ValueError(msg)


def gdn_status_string(status):
    return _lib.load().gdn_status_string(int(status)).decode()


def gdn_prefill_crossover_tokens(h_k, h_v, d_k, d_v, dtype=torch.bfloat16):
    return int(_lib.load().gdn_prefill_crossover_tokens(h_k, h_v, d_k, d_v, _DTYPES[dtype]))


def gdn_prefill_form(num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype=torch.bfloat16,
                     algo="auto", workspace_bytes=0, qk_l2norm=False, sm_count=0):
    """Name of the evaluation gdn_prefill would run for these sizes ("scan",
    "chunked_fused", "chunked_split" or "chunked_coop"; see gdn_prefill_form in
    include/gdn.h).  Raises GdnError for arguments the call would refuse."""
    r = int(_lib.load().gdn_prefill_form(num_seqs, total_tokens, h_k, h_v, d_k, d_v,
                                         _DTYPES[dtype], _lib.ALGOS[algo], int(workspace_bytes),
                                         _options(qk_l2norm), int(sm_count)))
    if r < 0:
        raise GdnError(-r, "gdn_prefill_form")
    return {v: k for k, v in _lib.ALGOS.items()}[r]


def gdn_prefill_workspace_size(num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype=torch.bfloat16,
                               algo="auto"):
    return int(_lib.load().gdn_prefill_workspace_size(num_seqs, total_tokens, h_k, h_v, d_k, d_v,
                                                      _DTYPES[dtype], _lib.ALGOS[algo]))


def _options(qk_l2norm):
    return _lib.GDN_OPT_QK_L2NORM if qk_l2norm else 0


def gdn_prefill(q, k, v, g, beta, cu_seqlens, state_in=None, state_out=None, o=None, scale=1.0,
                algo="auto", workspace=None, stream=None, qk_l2norm=False):
    """Prefill N packed sequences (see gdn_prefill in include/gdn.h).

    q, k [T, h_k, d_k]; v [T, h_v, d_v] (fp32 or bf16); g, beta [T, h_v] fp32;
    cu_seqlens [N+1] int32 on the device; state_in [N, h_v, d_v, d_k] fp32 or
    None (zeros).  Returns (o [T, h_v, d_v], state_out [N, h_v, d_v, d_k]).
    ``algo``: "auto", "scan", "chunked", "chunked_fused", "chunked_split" or "chunked_coop".
    ``qk_l2norm``: divide q and k by their per-head L2 norm inside the kernels.
    Without ``workspace`` one of the size gdn_prefill_workspace_size() reports
    is allocated (none when that is 0).
    """
    lib = _lib.load()
    T, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    _require(k.shape == q.shape and v.shape[0] == T, "q/k/v shapes disagree")
    _require(g.shape == (T, h_v) and beta.shape == (T, h_v), "g/beta must be [T, h_v]")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    _require(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda, "cu_seqlens: int32 on GPU")
    for t in (q, k, v, g, beta, cu_seqlens):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    _require(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share a dtype")
    if o is None:
        o = torch.empty((T, h_v, d_v), dtype=q.dtype, device=q.device)
    if state_out is None:
        state_out = torch.empty((N, h_v, d_v, d_k), dtype=torch.float32, device=q.device)
    if state_in is not None:
        _require(state_in.dtype == torch.float32 and state_in.is_contiguous(), "state_in fp32")
    need = lib.gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v, dt, _lib.ALGOS[algo])
    if qk_l2norm and algo in ("auto", "chunked"):
        # the normalisation option needs a workspace form (two kernels, or the
        # cooperative one when AUTO's size query already leaves room for it)
        need = max(need, lib.gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v, dt,
                                                        _lib.ALGOS["chunked_split"]))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.gdn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                            _ptr(state_out), _ptr(o), _ptr(cu_seqlens), N, T, h_k, h_v, d_k, d_v,
                            dt, float(scale), _lib.ALGOS[algo], _ptr(workspace), ws_bytes,
                            _options(qk_l2norm), _stream(stream))
    _lib.check(st, "gdn_prefill")
    return o, state_out


def gdn_prefill_streamed_workspace_size(piece_tokens, h_k, h_v, d_k, d_v, dtype=torch.bfloat16):
    return int(_lib.load().gdn_prefill_streamed_workspace_size(piece_tokens, h_k, h_v, d_k, d_v,
                                                               _DTYPES[dtype]))


def gdn_prefill_streamed(q, k, v, g, beta, piece_tokens, state_in=None, state_out=None, o=None,
                         scale=1.0, workspace=None, stream=None, qk_l2norm=False):
    """One sequence (q, k [T, h_k, d_k]; v [T, h_v, d_v]; g, beta [T, h_v]) prefilled
    as pieces of ``piece_tokens`` tokens (a multiple of 64) with the state carried
    between them (gdn_prefill_streamed in include/gdn.h).  Returns (o, state_out
    [1, h_v, d_v, d_k]); a workspace of gdn_prefill_streamed_workspace_size() bytes
    is allocated when none is given (its size does not depend on T)."""
    lib = _lib.load()
    T, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    _require(k.shape == q.shape and v.shape[0] == T, "q/k/v shapes disagree")
    _require(g.shape == (T, h_v) and beta.shape == (T, h_v), "g/beta must be [T, h_v]")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    for t in (q, k, v, g, beta):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((T, h_v, d_v), dtype=q.dtype, device=q.device)
    if state_out is None:
        state_out = torch.empty((1, h_v, d_v, d_k), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = lib.gdn_prefill_streamed_workspace_size(piece_tokens, h_k, h_v, d_k, d_v, dt)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_prefill_streamed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                                  _ptr(state_out), _ptr(o), T, h_k, h_v, d_k, d_v, dt,
                                  float(scale), int(piece_tokens), _ptr(workspace), ws_bytes,
                                  _options(qk_l2norm), _stream(stream))
    _lib.check(st, "gdn_prefill_streamed")
    return o, state_out


def gdn_prefill_host_workspace_size(piece_tokens, h_k, h_v, d_k, d_v, dtype=torch.bfloat16):
    return int(_lib.load().gdn_prefill_host_workspace_size(piece_tokens, h_k, h_v, d_k, d_v,
                                                           _DTYPES[dtype]))


def gdn_prefill_host(q, k, v, g, beta, piece_tokens=1024, state_in=None, state_out=None, o=None,
                     scale=1.0, workspace=None, stream=None, qk_l2norm=False, device=None):
    """gdn_prefill_host in include/gdn.h: one sequence whose tensors are on the HOST
    (q, k [T, h_k, d_k]; v [T, h_v, d_v]; g, beta [T, h_v]; page-locked for overlap),
    prefilled in pieces with the copies overlapped.  Outputs o [T, h_v, d_v] and
    state_out [1, h_v, d_v, d_k] are host tensors (page-locked ones are allocated
    when not given); a device workspace is allocated when none is given.  The
    results are ready once the stream is synchronised.  Returns (o, state_out)."""
    lib = _lib.load()
    T, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    _require(k.shape == q.shape and v.shape[0] == T, "q/k/v shapes disagree")
    _require(g.shape == (T, h_v) and beta.shape == (T, h_v), "g/beta must be [T, h_v]")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    for t in (q, k, v, g, beta, state_in):
        _require(t is None or (t.device.type == "cpu" and t.is_contiguous()),
                 "inputs must be contiguous host tensors")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((T, h_v, d_v), dtype=q.dtype).pin_memory()
    if state_out is None:
        state_out = torch.empty((1, h_v, d_v, d_k), dtype=torch.float32).pin_memory()
    _require(o.device.type == "cpu" and state_out.device.type == "cpu", "outputs must be on the host")
    if workspace is None:
        need = lib.gdn_prefill_host_workspace_size(piece_tokens, h_k, h_v, d_k, d_v, dt)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8,
                                device=device if device is not None else "cuda")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                              _ptr(state_out), _ptr(o), T, h_k, h_v, d_k, d_v, dt, float(scale),
                              int(piece_tokens), _ptr(workspace), ws_bytes, _options(qk_l2norm),
                              _stream(stream))
    _lib.check(st, "gdn_prefill_host")
    return o, state_out


def gdn_prefill_noalloc(q, k, v, g, beta, cu_seqlens, state_out, o, state_in=None, scale=1.0,
                        stream=None):
    """The two-kernel chunked prefill with the library's fixed scratch array
    (gdn_prefill_noalloc in include/gdn.h), for callers that cannot allocate
    device memory at call time.  Neither this wrapper nor the C entry point
    allocates: the caller passes every output (o [T, h_v, d_v] bf16,
    state_out [N, h_v, d_v, d_k] fp32).  Calls that overlap on the GPU race on
    the shared scratch; order them (e.g. on one stream)."""
    lib = _lib.load()
    T, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    _require(k.shape == q.shape and v.shape[0] == T, "q/k/v shapes disagree")
    _require(g.shape == (T, h_v) and beta.shape == (T, h_v), "g/beta must be [T, h_v]")
    _require(o.shape == (T, h_v, d_v) and state_out.shape == (N, h_v, d_v, d_k),
             "o / state_out shapes")
    for t in (q, k, v, g, beta, cu_seqlens, o, state_out):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    st = lib.gdn_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                                 _ptr(state_out), _ptr(o), _ptr(cu_seqlens), N, T, h_k, h_v, d_k,
                                 d_v, dt, float(scale), _stream(stream))
    _lib.check(st, "gdn_prefill_noalloc")
    return o, state_out


def gdn_decode_step(q, k, v, g, beta, state, o=None, scale=1.0, stream=None, qk_l2norm=False):
    """One token per sequence, state [B, h_v, d_v, d_k] fp32 updated in place.

    q, k [B, h_k, d_k]; v [B, h_v, d_v]; g, beta [B, h_v] fp32.  Returns o [B, h_v, d_v].
    """
    lib = _lib.load()
    B, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    _require(k.shape == q.shape and v.shape[0] == B, "q/k/v shapes disagree")
    _require(state.shape == (B, h_v, d_v, d_k) and state.dtype == torch.float32,
             "state must be [B, h_v, d_v, d_k] fp32")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    for t in (q, k, v, g, beta, state):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((B, h_v, d_v), dtype=q.dtype, device=q.device)
    st = lib.gdn_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                _ptr(o), B, h_k, h_v, d_k, d_v, dt, float(scale),
                                _options(qk_l2norm), _stream(stream))
    _lib.check(st, "gdn_decode_step")
    return o


def gdn_decode_step_rmsnorm(q, k, v, g, beta, state, norm_weight=None, norm_eps=1e-6, o=None,
                            scale=1.0, stream=None, qk_l2norm=False):
    """gdn_decode_step with the output RMS-normalised in the same kernel
    (gdn_decode_step_rmsnorm in include/gdn.h): o[b, h] = w * y / rms(y) over the
    d_v values, norm_weight [d_v] fp32 or None (ones)."""
    lib = _lib.load()
    B, h_k, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    _require(k.shape == q.shape and v.shape[0] == B, "q/k/v shapes disagree")
    _require(state.shape == (B, h_v, d_v, d_k) and state.dtype == torch.float32,
             "state must be [B, h_v, d_v, d_k] fp32")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    if norm_weight is not None:
        _require(norm_weight.shape == (d_v,) and norm_weight.dtype == torch.float32,
                 "norm_weight must be [d_v] fp32")
    for t in (q, k, v, g, beta, state, norm_weight):
        _require(t is None or t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((B, h_v, d_v), dtype=q.dtype, device=q.device)
    st = lib.gdn_decode_step_rmsnorm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                     _ptr(o), _ptr(norm_weight), float(norm_eps), B, h_k, h_v,
                                     d_k, d_v, dt, float(scale), _options(qk_l2norm),
                                     _stream(stream))
    _lib.check(st, "gdn_decode_step_rmsnorm")
    return o


def gdn_output_rmsnorm(o, norm_weight=None, norm_eps=1e-6, stream=None):
    """The output RMS normalisation in place over o [..., h_v, d_v] (gdn_output_rmsnorm
    in include/gdn.h); returns o."""
    lib = _lib.load()
    _require(o.dim() >= 2 and o.is_contiguous(), "o must be contiguous [..., h_v, d_v]")
    h_v, d_v = o.shape[-2], o.shape[-1]
    rows = o.numel() // (h_v * d_v) if o.numel() else 0
    if norm_weight is not None:
        _require(norm_weight.shape == (d_v,) and norm_weight.dtype == torch.float32 and
                 norm_weight.is_contiguous(), "norm_weight must be [d_v] fp32")
    st = lib.gdn_output_rmsnorm(_ptr(o), _ptr(norm_weight), rows, h_v, d_v, _dtype_code(o),
                                float(norm_eps), _stream(stream))
    _lib.check(st, "gdn_output_rmsnorm")
    return o


def gdn_decode_multi(q, k, v, g, beta, state, o=None, snapshots=False, scale=1.0, stream=None,
                     qk_l2norm=False):
    """n tokens for each of B sequences in one launch (gdn_decode_multi in
    include/gdn.h): q, k [B, n, h_k, d_k]; v [B, n, h_v, d_v]; g, beta [B, n, h_v]
    fp32; state [B, h_v, d_v, d_k] fp32 updated in place to the state after the
    last token.  ``snapshots``: False (none), True (allocated and returned) or a
    [B, n, h_v, d_v, d_k] fp32 tensor receiving the state after each token.
    Returns o [B, n, h_v, d_v], or (o, snapshots) when snapshots are asked for."""
    lib = _lib.load()
    B, n, h_k, d_k = q.shape
    h_v, d_v = v.shape[2], v.shape[3]
    _require(k.shape == q.shape and v.shape[:2] == (B, n), "q/k/v shapes disagree")
    _require(g.shape == (B, n, h_v) and beta.shape == (B, n, h_v), "g/beta must be [B, n, h_v]")
    _require(state.shape == (B, h_v, d_v, d_k) and state.dtype == torch.float32,
             "state must be [B, h_v, d_v, d_k] fp32")
    _require(g.dtype == torch.float32 and beta.dtype == torch.float32, "g/beta must be fp32")
    for t in (q, k, v, g, beta, state):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((B, n, h_v, d_v), dtype=q.dtype, device=q.device)
    snap = None
    if snapshots is True:
        snap = torch.empty((B, n, h_v, d_v, d_k), dtype=torch.float32, device=q.device)
    elif snapshots is not False and snapshots is not None:
        snap = snapshots
        _require(snap.shape == (B, n, h_v, d_v, d_k) and snap.dtype == torch.float32 and
                 snap.is_contiguous(), "snapshots must be [B, n, h_v, d_v, d_k] fp32")
    st = lib.gdn_decode_multi(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                              _ptr(o), _ptr(snap), B, n, h_k, h_v, d_k, d_v, dt, float(scale),
                              _options(qk_l2norm), _stream(stream))
    _lib.check(st, "gdn_decode_multi")
    return o if snap is None else (o, snap)


def gdn_attn_decode_workspace_size(batch, h_q, h_kv, head_dim, capacity, layout="auto",
                                   block_keys=0):
    return int(_lib.load().gdn_attn_decode_workspace_size(batch, h_q, h_kv, head_dim, capacity,
                                                          _lib.ATTN_LAYOUTS[layout],
                                                          int(block_keys)))


def gdn_attn_decode_block_keys(batch, h_q, h_kv, head_dim, capacity, layout="auto",
                               block_keys=0):
    """Keys per CTA block that gdn_attn_decode would use on the current device (-1 if invalid)."""
    return int(_lib.load().gdn_attn_decode_block_keys(batch, h_q, h_kv, head_dim, capacity,
                                                      _lib.ATTN_LAYOUTS[layout],
                                                      int(block_keys)))


def gdn_attn_decode(q, k_cache, v_cache, cache_len, scale=None, o=None, layout="auto",
                    block_keys=0, workspace=None, stream=None):
    """Grouped-query decode attention (gdn_attn_decode in include/gdn.h): q
    [B, h_q, D]; k_cache, v_cache [B, h_kv, capacity, D]; cache_len [B] int32 on
    the device; all bf16, D = 256, h_q / h_kv <= 8.  ``scale`` defaults to
    1/sqrt(D).  ``layout``: "auto", "general" or "fixed_block" (blocks of
    ``block_keys`` keys, 0 = the library's choice).  A workspace of
    gdn_attn_decode_workspace_size() bytes is allocated when none is given and
    the layout may need one.  Returns o [B, h_q, D]."""
    lib = _lib.load()
    B, h_q, D = q.shape
    h_kv, cap = k_cache.shape[1], k_cache.shape[2]
    _require(k_cache.shape == (B, h_kv, cap, D) and v_cache.shape == k_cache.shape,
             "k_cache / v_cache must be [B, h_kv, capacity, D]")
    _require(cache_len.shape == (B,) and cache_len.dtype == torch.int32,
             "cache_len must be [B] int32")
    for t in (q, k_cache, v_cache, cache_len):
        _require(t.is_contiguous(), "tensors must be contiguous")
    dt = _dtype_code(q)
    if scale is None:
        scale = D ** -0.5
    if o is None:
        o = torch.empty((B, h_q, D), dtype=q.dtype, device=q.device)
    lay = _lib.ATTN_LAYOUTS[layout]
    if workspace is None and layout != "general":
        need = lib.gdn_attn_decode_workspace_size(B, h_q, h_kv, D, cap, lay, int(block_keys))
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.gdn_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), _ptr(o), B,
                             h_q, h_kv, D, cap, dt, float(scale), lay, int(block_keys),
                             _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check(st, "gdn_attn_decode")
    return o


def gdn_stream_status(stream=None):
    """Synchronise the stream; return (and clear) the device error word as a status name."""
    return STATUS_NAMES.get(int(_lib.load().gdn_stream_status(_stream(stream))), "unknown")


def gdn_selftest_wait_timeout(timeout_us=1000, stream=None):
    """Enqueue the bounded-wait self-test (see gdn_selftest_wait_timeout in
    include/gdn.h): a device wait that expires and records GDN_ERR_DEVICE_TIMEOUT,
    which the next gdn_stream_status reports."""
    _lib.check(_lib.load().gdn_selftest_wait_timeout(int(timeout_us), _stream(stream)),
               "gdn_selftest_wait_timeout")
