"""Python binding of the TwoTower block-diffusion denoise-step library (libtdenoise.so).

Argument marshalling only: every step of the path runs in the CUDA kernels behind the C ABI
declared in include/td.h. PyTorch supplies device memory and streams. There is no CPU
fallback: if the library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtdenoise.so")

TD_FN_ADALN_MODULATE = 0
TD_FN_BLOCK_ATTENTION = 1
TD_FN_LMHEAD_COMMIT = 2
TD_FN_DENOISE_STEP = 3
TD_FN_DECODE_BLOCK = 4

TD_COMMIT_CONFIDENCE = 0      # mask-diffusion: confidence masking with threshold gamma
TD_COMMIT_LEFT_TO_RIGHT = 1   # mock-AR reading: one commit per step, lowest masked index

TD_ATTN_P_BF16 = 0    # attention probabilities rounded to bf16 for the P V product (default)
TD_ATTN_P_SPLIT = 1   # carried as a hi + lo pair of bf16 values (a second P V product)

# Every symbol the header declares (checked by the tests).
EXPORTED = ("td_workspace_size", "td_status_string", "td_adaln_modulate", "td_block_attention",
            "td_lmhead_commit", "td_denoise_step", "td_decode_block", "td_device_error",
            "td_lmhead_commit_static", "td_kv_append", "td_check_bounded_wait",
            "td_timestep_table", "td_decode_graph_form")


class TdError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


class td_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "S", "d", "Hq", "Hkv", "D", "V", "Lmax",
                                             "n_layers")]


class td_layer(ctypes.Structure):
    _fields_ = [("wqkv", ctypes.c_void_p), ("wo", ctypes.c_void_p), ("ada_E", ctypes.c_void_p),
                ("k_ctx", ctypes.c_void_p), ("v_ctx", ctypes.c_void_p)]


class td_paging(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("max_pages", ctypes.c_int),
                ("n_pages", ctypes.c_int)]


class td_step_opts(ctypes.Structure):
    _fields_ = [("rule", ctypes.c_int), ("rope_theta", ctypes.c_float), ("paging", td_paging),
                ("h_out", ctypes.c_void_p), ("attn_precision", ctypes.c_int)]


class td_kv(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m block_diffusion_lm_denoise_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.td_workspace_size.argtypes = [ctypes.POINTER(td_dims), i]
        L.td_workspace_size.restype = sz
        L.td_status_string.argtypes = [i]
        L.td_status_string.restype = ctypes.c_char_p
        L.td_adaln_modulate.argtypes = [vp, vp, vp, i, i, f, vp, vp]
        L.td_block_attention.argtypes = [ctypes.POINTER(td_dims), vp, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(td_paging), i, vp, vp, vp, sz, vp]
        L.td_lmhead_commit.argtypes = [ctypes.POINTER(td_dims), vp, vp, f, i, i, vp, vp, vp, vp,
                                       vp, vp, vp, sz, vp]
        L.td_denoise_step.argtypes = [ctypes.POINTER(td_dims), ctypes.POINTER(td_layer), vp, vp,
                                      vp, vp, vp, vp, i, i, f, ctypes.POINTER(td_step_opts), vp,
                                      vp, vp, vp, vp, vp, vp, sz, vp]
        L.td_decode_block.argtypes = [ctypes.POINTER(td_dims), ctypes.POINTER(td_layer), vp, vp,
                                      vp, vp, vp, i, i, f, ctypes.POINTER(td_step_opts), vp, vp,
                                      vp, vp, vp, vp, ctypes.POINTER(i), vp, sz, vp]
        L.td_kv_append.argtypes = [ctypes.POINTER(td_dims), ctypes.POINTER(td_layer),
                                   ctypes.POINTER(td_kv), vp, ctypes.POINTER(td_paging), vp]
        L.td_device_error.argtypes = [ctypes.POINTER(i)]
        L.td_check_bounded_wait.argtypes = [ctypes.c_uint, vp]
        L.td_timestep_table.argtypes = [vp, vp, i, i, vp, vp]
        L.td_decode_graph_form.argtypes = [i]
        L.td_lmhead_commit_static.argtypes = [ctypes.POINTER(td_dims), vp, vp, f, i, vp, vp, vp,
                                               vp, vp, vp, vp]
        for name in EXPORTED:
            if name not in ("td_workspace_size", "td_status_string"):
                getattr(L, name).restype = i
        _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise TdError(fn, status, lib().td_status_string(status).decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_dims(B, S, d, Hq, Hkv, D, V, Lmax, n_layers) -> td_dims:
    """td_dims from its nine sizes (sequences, block size, hidden size, query / KV heads,
    head dim, vocabulary, context capacity, layers)."""
    return td_dims(B, S, d, Hq, Hkv, D, V, Lmax, n_layers)


def dims_from(obj) -> td_dims:
    """td_dims from a mapping or an object with the nine fields."""
    get = (lambda k: obj[k]) if isinstance(obj, dict) else (lambda k: getattr(obj, k))
    return td_dims(*(int(get(k)) for k in ("B", "S", "d", "Hq", "Hkv", "D", "V", "Lmax",
                                          "n_layers")))


def td_workspace_size(dims, fn: int) -> int:
    """Bytes of caller workspace entry point `fn` (a TD_FN_* value) needs at these sizes;
    raises TdError for sizes the kernels do not support."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    n = lib().td_workspace_size(ctypes.byref(dm), fn)
    if n == ctypes.c_size_t(-1).value:
        raise TdError("td_workspace_size", 3, "unsupported or invalid dims")
    return int(n)


def workspace(dims, fn: int, device="cuda") -> torch.Tensor:
    """A device byte buffer of td_workspace_size(dims, fn) bytes (at least 256)."""
    return torch.empty(max(256, td_workspace_size(dims, fn)), dtype=torch.uint8, device=device)


def td_device_error() -> int:
    """Reads and clears the device error word (0 = none). A wait code (0x100, 0x200,
    0x300) comes back as the library's TD_ERR_DEVICE_TIMEOUT status, returned here as the
    code itself."""
    code = ctypes.c_int(0)
    st = lib().td_device_error(ctypes.byref(code))
    if st not in (0, 6):
        _check("td_device_error", st)
    return code.value


def td_adaln_modulate(h: torch.Tensor, E: torch.Tensor, phi: torch.Tensor, eps: float = 1e-6,
                      x_mod: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x_mod = bf16(LayerNorm(h) * (1 + m[1]) + m[0]) with m = E + phi, for h bf16 [rows, d]
    and E, phi fp32 [6, d]; returns x_mod (allocated when not given)."""
    rows, d = h.shape
    if x_mod is None:
        x_mod = torch.empty_like(h)
    _check("td_adaln_modulate",
           lib().td_adaln_modulate(_ptr(h), _ptr(E), _ptr(phi), rows, d, eps, _ptr(x_mod),
                                   _stream(stream)))
    return x_mod


def _paging(page_table, n_pages):
    """td_paging for a page table [B, max_pages] (int32 device tensor) or None."""
    if page_table is None:
        return None
    return td_paging(_ptr(page_table), int(page_table.shape[1]), int(n_pages))


def td_block_attention(dims, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len=None, o=None, lse=None,
                       ws=None, stream=None, page_table=None, n_pages=0,
                       precision: int = TD_ATTN_P_BF16):
    """page_table [B, max_pages] int32 with k_ctx / v_ctx as page pools [n_pages, Hkv, 128, D]
    selects the paged layout; precision: TD_ATTN_P_BF16 or TD_ATTN_P_SPLIT."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    if o is None:
        o = torch.empty_like(q)
    if ws is None:
        ws = workspace(dm, TD_FN_BLOCK_ATTENTION, q.device)
    _check("td_block_attention",
           lib().td_block_attention(ctypes.byref(dm), _ptr(q), _ptr(k_blk), _ptr(v_blk),
                                    _ptr(k_ctx), _ptr(v_ctx), _ptr(ctx_len),
                                    _byref_or_null(_paging(page_table, n_pages)),
                                    int(precision), _ptr(o),
                                    _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return o


def _byref_or_null(x):
    return None if x is None else ctypes.byref(x)


def _opts(rule, rope_theta, page_table, n_pages, h_out=None, attn_precision=0):
    pg = _paging(page_table, n_pages)
    return td_step_opts(int(rule), float(rope_theta), pg if pg is not None else td_paging(),
                        _ptr(h_out), int(attn_precision))


def _outs(B, S, device, conf, pred, n_committed, all_done):
    if conf is None:
        conf = torch.empty((B, S), dtype=torch.float32, device=device)
    if pred is None:
        pred = torch.empty((B, S), dtype=torch.int32, device=device)
    if n_committed is None:
        n_committed = torch.empty((B,), dtype=torch.int32, device=device)
    if all_done is None:
        all_done = torch.empty((1,), dtype=torch.int32, device=device)
    return conf, pred, n_committed, all_done


def td_lmhead_commit(dims, h, w_lm, gamma: float, force_all: bool, tokens, masked, conf=None,
                     pred=None, n_committed=None, all_done=None, ws=None, stream=None,
                     rule: int = TD_COMMIT_CONFIDENCE):
    """Updates tokens / masked in place; returns (conf, pred, n_committed, all_done)."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    conf, pred, n_committed, all_done = _outs(dm.B, dm.S, h.device, conf, pred, n_committed,
                                              all_done)
    if ws is None:
        ws = workspace(dm, TD_FN_LMHEAD_COMMIT, h.device)
    _check("td_lmhead_commit",
           lib().td_lmhead_commit(ctypes.byref(dm), _ptr(h), _ptr(w_lm), gamma, int(rule),
                                  int(force_all),
                                  _ptr(tokens), _ptr(masked), _ptr(conf), _ptr(pred),
                                  _ptr(n_committed), _ptr(all_done), _ptr(ws), ws.numel(),
                                  _stream(stream)))
    return conf, pred, n_committed, all_done


def td_lmhead_commit_static(dims, h, w_lm, gamma: float, force_all: bool, tokens, masked,
                            conf=None, pred=None, n_committed=None, all_done=None, stream=None):
    """td_lmhead_commit with the library's fixed 16 MiB device scratch instead of a
    caller workspace (for callers that cannot allocate); calls must not overlap on the GPU."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    conf, pred, n_committed, all_done = _outs(dm.B, dm.S, h.device, conf, pred, n_committed,
                                              all_done)
    _check("td_lmhead_commit_static",
           lib().td_lmhead_commit_static(ctypes.byref(dm), _ptr(h), _ptr(w_lm), gamma,
                                         int(force_all), _ptr(tokens), _ptr(masked), _ptr(conf),
                                         _ptr(pred), _ptr(n_committed), _ptr(all_done),
                                         _stream(stream)))
    return conf, pred, n_committed, all_done


def _layers(layers: Sequence[Dict[str, torch.Tensor]]):
    arr = (td_layer * max(1, len(layers)))()
    for i, L in enumerate(layers):
        arr[i] = td_layer(_ptr(L["wqkv"]), _ptr(L["wo"]), _ptr(L["ada_E"]),
                          _ptr(L.get("k_ctx")), _ptr(L.get("v_ctx")))
    return arr


def td_denoise_step(dims, layers, w_lm, phi_t, t: int, T: int, gamma: float, tokens, masked,
                    h=None, emb=None, pos=None, ctx_len=None, conf=None, pred=None,
                    n_committed=None, all_done=None, ws=None, stream=None,
                    rule: int = TD_COMMIT_CONFIDENCE, rope_theta: float = 0.0,
                    page_table=None, n_pages: int = 0, h_out=None,
                    attn_precision: int = TD_ATTN_P_BF16):
    """One denoising step; tokens / masked updated in place.
    rule: commit rule; rope_theta > 0: rotary variant (see td_step_opts in include/td.h);
    h_out (bf16 [B*S, d] device tensor): receives the hidden state after the last layer;
    attn_precision: TD_ATTN_P_BF16 or TD_ATTN_P_SPLIT.
    Returns (conf, pred, n_committed, all_done)."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    dev = w_lm.device
    conf, pred, n_committed, all_done = _outs(dm.B, dm.S, dev, conf, pred, n_committed,
                                              all_done)
    if ws is None:
        ws = workspace(dm, TD_FN_DENOISE_STEP, dev)
    arr = _layers(layers)
    _check("td_denoise_step",
           lib().td_denoise_step(ctypes.byref(dm), arr, _ptr(ctx_len), _ptr(h), _ptr(emb),
                                 _ptr(pos), _ptr(w_lm), _ptr(phi_t), t, T, gamma,
                                 ctypes.byref(_opts(rule, rope_theta, page_table, n_pages,
                                                    h_out, attn_precision)),
                                 _ptr(tokens),
                                 _ptr(masked), _ptr(conf), _ptr(pred), _ptr(n_committed),
                                 _ptr(all_done), _ptr(ws), ws.numel(), _stream(stream)))
    return conf, pred, n_committed, all_done


def td_decode_block(dims, layers, emb, pos, w_lm, phi_table, T: int, gamma: float, tokens,
                    masked, t_start: int = 1, ctx_len=None, conf=None, pred=None,
                    n_committed=None, all_done=None, ws=None, stream=None,
                    rule: int = TD_COMMIT_CONFIDENCE, rope_theta: float = 0.0,
                    page_table=None, n_pages: int = 0,
                    attn_precision: int = TD_ATTN_P_BF16) -> int:
    """Runs the block decode loop in place on tokens / masked; returns the steps taken."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    dev = w_lm.device
    conf, pred, n_committed, all_done = _outs(dm.B, dm.S, dev, conf, pred, n_committed,
                                              all_done)
    if ws is None:
        ws = workspace(dm, TD_FN_DECODE_BLOCK, dev)
    steps = ctypes.c_int(0)
    arr = _layers(layers)
    _check("td_decode_block",
           lib().td_decode_block(ctypes.byref(dm), arr, _ptr(ctx_len), _ptr(emb), _ptr(pos),
                                 _ptr(w_lm), _ptr(phi_table), t_start, T, gamma,
                                 ctypes.byref(_opts(rule, rope_theta, page_table, n_pages,
                                                    None, attn_precision)),
                                 _ptr(tokens),
                                 _ptr(masked), _ptr(conf), _ptr(pred), _ptr(n_committed),
                                 _ptr(all_done), ctypes.byref(steps), _ptr(ws), ws.numel(),
                                 _stream(stream)))
    return steps.value


def td_kv_append(dims, layers, block_kv, ctx_len, stream=None, page_table=None,
                 n_pages: int = 0) -> None:
    """Appends each layer's committed-block keys / values (block_kv: a list of (k, v) device
    tensors [B, S, Hkv, D] bf16) to that layer's context cache at ctx_len, and grows
    ctx_len [B] (int32, device) by S, on the device."""
    dm = dims if isinstance(dims, td_dims) else dims_from(dims)
    arr = _layers(layers)
    kv = (td_kv * max(1, len(block_kv)))()
    for i, (k, v) in enumerate(block_kv):
        kv[i] = td_kv(_ptr(k), _ptr(v))
    _check("td_kv_append", lib().td_kv_append(ctypes.byref(dm), arr, kv, _ptr(ctx_len),
                                              _byref_or_null(_paging(page_table, n_pages)),
                                              _stream(stream)))


def td_check_bounded_wait(limit_us: int, stream=None) -> None:
    """Launches the bounded-wait diagnostic (see include/td.h); read the result with
    td_device_error()."""
    _check("td_check_bounded_wait", lib().td_check_bounded_wait(int(limit_us), _stream(stream)))


TD_GRAPH_CONDITIONAL = 1   # decode-loop graph: one conditional node per step
TD_GRAPH_FLAT = 2          # decode-loop graph: one flat capture, finished steps return at once


def td_decode_graph_form(form: int = 0) -> int:
    """Diagnostic (see include/td.h): form 1 or 2 selects the form of decode-loop graphs built
    from now on; returns the form of the last graph built (0 before the first)."""
    return int(lib().td_decode_graph_form(int(form)))


def td_timestep_table(w_t, b_t, T: int, phi_table=None, stream=None) -> torch.Tensor:
    """The adaLN-single table phi(t), t = 1..T, fp32 [T, 6, d], from W_t fp32 [6d, 256] and
    b_t fp32 [6d] (see include/td.h); allocated when not given."""
    d = int(b_t.numel()) // 6
    if phi_table is None:
        phi_table = torch.empty((T, 6, d), dtype=torch.float32, device=b_t.device)
    _check("td_timestep_table", lib().td_timestep_table(_ptr(w_t), _ptr(b_t), d, int(T),
                                                        _ptr(phi_table), _stream(stream)))
    return phi_table
