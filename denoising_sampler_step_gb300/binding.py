"""Python binding of libdgsamp: argument marshalling only.

Every function here has the name of the C entry point it calls (include/dgsamp.h)
and does nothing but turn torch CUDA tensors into pointers, sizes and the current
stream, allocate outputs with torch when the caller gives none, and raise on a
non-zero status.  All arithmetic runs in the library's CUDA kernels; there is no
other path.  Importing this module fails if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdgsamp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m denoising_sampler_step_gb300.build` "
        "(or __graft_entry__.build()); there is no fallback path")

lib = ctypes.CDLL(LIB_PATH)

_i64, _i32, _f32, _p, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_u32 = ctypes.c_uint32

# flags of the sampler-step calls (dg_step_flags)
DG_STEP_TWO_PASS = 1

lib.dg_version.restype = ctypes.c_int
lib.dg_last_error.restype = ctypes.c_char_p
lib.dg_row_stats.argtypes = [_p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p]
lib.dg_row_stats.restype = ctypes.c_int
lib.dg_soft_embed_workspace_size.argtypes = [_i64, _i64, _i64]
lib.dg_soft_embed_workspace_size.restype = _sz
lib.dg_soft_embed.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _i64, _i64, _f32, _p, _i64, _p, _sz, _p]
lib.dg_soft_embed.restype = ctypes.c_int
lib.dg_soft_embed_no_alloc.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _i64, _i64, _f32, _p, _i64, _p]
lib.dg_soft_embed_no_alloc.restype = ctypes.c_int
lib.dg_entropy_accept.argtypes = [_p, _p, _i32, _i32, _p, _i32, _p, _p, _p, _p]
lib.dg_entropy_accept.restype = ctypes.c_int
lib.dg_sum_partials.argtypes = [ctypes.POINTER(_p), _i32, _i64, _i64, _i64, _f32, _p, _i64, _p]
lib.dg_sum_partials.restype = ctypes.c_int
lib.dg_sampler_step.argtypes = [_p, _i32, _i32, _i64, _i64, _p, _i64, _i64, _i64, _i64, _i64, _f32, _p, _i32,
                                _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _u32, _p, _sz, _p]
lib.dg_sampler_step.restype = ctypes.c_int
lib.dg_get_device_status.argtypes = [_p]
lib.dg_get_device_status.restype = ctypes.c_int
lib.dg_row_sample.argtypes = [_p, _i64, _i64, _i64, _f32, ctypes.c_uint64, ctypes.c_uint64, _p, _p, _p]
lib.dg_row_sample.restype = ctypes.c_int
lib.dg_check_wait_timeout.argtypes = [ctypes.c_uint32, _p]
lib.dg_check_wait_timeout.restype = ctypes.c_int
lib.dg_entropy_accept_eligible.argtypes = [_p, _p, _p, _i32, _i32, _p, _i32, _p, _p, _p, _p]
lib.dg_entropy_accept_eligible.restype = ctypes.c_int
lib.dg_loop_update.argtypes = [_p, _p, _p, _p, _i32, _i32, _i32, _f32, _i32, _p, _p, _p, _p, _p, _p, _p]
lib.dg_loop_update.restype = ctypes.c_int
lib.dg_sampler_loop_step.argtypes = [_p, _i32, _i32, _i64, _i64, _p, _i64, _i64, _i64, _i64, _i64, _f32, _p, _i32,
                                     _i32, _f32, _i32, _f32, ctypes.c_uint64, ctypes.c_uint64,
                                     _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64,
                                     _p, _p, _p, _p, _p, _p, _u32, _p, _sz, _p]
lib.dg_row_stats_sample.argtypes = [_p, _i64, _i64, _i64, _f32, ctypes.c_uint64, ctypes.c_uint64,
                                    _p, _p, _p, _p, _p, _p, _p, _p]
lib.dg_row_stats_sample.restype = ctypes.c_int
lib.dg_row_stats_partial.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _p]
lib.dg_row_stats_partial.restype = ctypes.c_int
lib.dg_row_stats_combine.argtypes = [_p, _i32, _i64, _p, _p, _p, _p, _p, _p]
lib.dg_row_stats_combine.restype = ctypes.c_int
lib.dg_sampler_loop_step.restype = ctypes.c_int
lib.dg_quantize_e4m3.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.dg_quantize_e4m3.restype = ctypes.c_int
lib.dg_soft_embed_workspace_size_e4m3.argtypes = [_i64, _i64, _i64]
lib.dg_soft_embed_workspace_size_e4m3.restype = _sz
lib.dg_soft_embed_e4m3.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _i64, _f32, _p, _i64, _p,
                                   _sz, _p]
lib.dg_soft_embed_e4m3.restype = ctypes.c_int
lib.dg_sampler_step_e4m3.argtypes = [_p, _i32, _i32, _i64, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64, _f32, _p,
                                     _i32, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _u32, _p, _sz, _p]
lib.dg_sampler_step_e4m3.restype = ctypes.c_int
lib.dg_sampler_loop_step_e4m3.argtypes = [_p, _i32, _i32, _i64, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64, _f32, _p,
                                          _i32, _i32, _f32, _i32, _f32, ctypes.c_uint64, ctypes.c_uint64,
                                          _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64,
                                          _p, _p, _p, _p, _p, _p, _u32, _p, _sz, _p]
lib.dg_sampler_loop_step_e4m3.restype = ctypes.c_int
lib.dg_soft_embed_shard_begin.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64, _i64, _i64, _p, _p, _sz, _p]
lib.dg_soft_embed_shard_begin.restype = ctypes.c_int
lib.dg_soft_embed_shard_end.argtypes = [_p, _i64, _p, _i64, _i64, _p, _i64, _i64, _i64, _f32, _p, _i64, _p, _sz, _p]
lib.dg_soft_embed_shard_end.restype = ctypes.c_int
lib.dg_soft_embed_shard_begin_e4m3.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]
lib.dg_soft_embed_shard_begin_e4m3.restype = ctypes.c_int
lib.dg_soft_embed_shard_end_e4m3.argtypes = [_p, _i64, _p, _i64, _i64, _p, _p, _i64, _i64, _i64, _f32, _p, _i64, _p,
                                             _sz, _p]
lib.dg_soft_embed_shard_end_e4m3.restype = ctypes.c_int

STATUS = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED", 3: "DG_ERR_CUDA", 4: "DG_ERR_TIMEOUT"}


class DgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.dg_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DgError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def _flags(two_pass: bool) -> int:
    return DG_STEP_TWO_PASS if two_pass else 0


def _new(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def dg_row_stats(logits: torch.Tensor, V: int | None = None, stream=None, out: dict | None = None) -> dict:
    """Row statistics of fp32 logits [R, >=V] -> dict m, lse, H, kappa (fp32), argmax (int32)."""
    R = logits.shape[0]
    V = logits.shape[1] if V is None else V
    dev = logits.device
    o = out
    if o is None:
        o = {k: _new(R, torch.float32, dev) for k in ("m", "lse", "H", "kappa")}
        o["argmax"] = _new(R, torch.int32, dev)
    _check(lib.dg_row_stats(_ptr(logits), R, V, _ld(logits), _ptr(o["m"]), _ptr(o["lse"]), _ptr(o["H"]),
                            _ptr(o["kappa"]), _ptr(o["argmax"]), _stream(stream)), "dg_row_stats")
    return o


def dg_row_sample(logits: torch.Tensor, temperature: float = 1.0, seed: int = 0, offset: int = 0,
                  V: int | None = None, stream=None, out: dict | None = None) -> dict:
    """Gumbel-max candidate per row of fp32 logits [R, >=V] at `temperature`, uniforms from
    Philox4x32-10 keyed by `seed` at step `offset` -> dict candidate (int32), log_p (fp32)."""
    R = logits.shape[0]
    V = logits.shape[1] if V is None else V
    dev = logits.device
    o = out
    if o is None:
        o = {"candidate": _new(R, torch.int32, dev), "log_p": _new(R, torch.float32, dev)}
    _check(lib.dg_row_sample(_ptr(logits), R, V, _ld(logits), float(temperature), int(seed), int(offset),
                             _ptr(o["candidate"]), _ptr(o["log_p"]), _stream(stream)), "dg_row_sample")
    return o


def dg_row_stats_partial(shard: torch.Tensor, vocab_offset: int, n: int | None = None, stream=None,
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """The shard's 16-byte summary per row: a [R, 4] float32 tensor whose column 1 holds the
    int32 bits of the global argmax (view it with .view(torch.int32))."""
    R = shard.shape[0]
    n = shard.shape[1] if n is None else n
    o = out if out is not None else _new((R, 4), torch.float32, shard.device)
    _check(lib.dg_row_stats_partial(_ptr(shard), R, n, _ld(shard), vocab_offset, _ptr(o), _stream(stream)),
           "dg_row_stats_partial")
    return o


def dg_soft_embed_shard_begin(shard: torch.Tensor, vocab_offset: int, W_shard, ws: torch.Tensor,
                              stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """First call of a shard's one-read soft embedding: the shard's [R, 4] row summaries (the
    format of dg_row_stats_partial); the split partials stay in `ws` for dg_soft_embed_shard_end.
    W_shard: bf16 [rows_pad, >= d], or an 8-bit table (codes, row scales)."""
    R, n = shard.shape
    o = out if out is not None else _new((R, 4), torch.float32, shard.device)
    if isinstance(W_shard, tuple):
        Q, scale = W_shard
        _check(lib.dg_soft_embed_shard_begin_e4m3(_ptr(shard), _ld(shard), R, n, vocab_offset, _ptr(Q), _ptr(scale),
                                                  Q.shape[0], _ld(Q), Q.shape[1], _ptr(o), _ptr(ws), ws.numel(),
                                                  _stream(stream)), "dg_soft_embed_shard_begin_e4m3")
    else:
        _check(lib.dg_soft_embed_shard_begin(_ptr(shard), _ld(shard), R, n, vocab_offset, _ptr(W_shard),
                                             W_shard.shape[0], _ld(W_shard), W_shard.shape[1], _ptr(o), _ptr(ws),
                                             ws.numel(), _stream(stream)), "dg_soft_embed_shard_begin")
    return o


def dg_soft_embed_shard_end(shard: torch.Tensor, lse: torch.Tensor, W_shard, gamma: float, ws: torch.Tensor,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Second call: gamma * E_shard [R, d] from the partials the first call left in `ws`, scaled
    against the full-row lse."""
    R, n = shard.shape
    d = W_shard[0].shape[1] if isinstance(W_shard, tuple) else W_shard.shape[1]
    if out is None:
        out = _new((R, d), torch.float32, shard.device)
    if isinstance(W_shard, tuple):
        Q, scale = W_shard
        _check(lib.dg_soft_embed_shard_end_e4m3(_ptr(shard), _ld(shard), _ptr(lse), R, n, _ptr(Q), _ptr(scale),
                                                Q.shape[0], _ld(Q), d, gamma, _ptr(out), _ld(out), _ptr(ws),
                                                ws.numel(), _stream(stream)), "dg_soft_embed_shard_end_e4m3")
    else:
        _check(lib.dg_soft_embed_shard_end(_ptr(shard), _ld(shard), _ptr(lse), R, n, _ptr(W_shard),
                                           W_shard.shape[0], _ld(W_shard), d, gamma, _ptr(out), _ld(out), _ptr(ws),
                                           ws.numel(), _stream(stream)), "dg_soft_embed_shard_end")
    return out


def dg_soft_embed_shard_begin_e4m3(shard: torch.Tensor, vocab_offset: int, Q_shard: torch.Tensor,
                                   scale_shard: torch.Tensor, ws: torch.Tensor, stream=None,
                                   out: torch.Tensor | None = None) -> torch.Tensor:
    """dg_soft_embed_shard_begin over an 8-bit table shard (codes, row scales)."""
    return dg_soft_embed_shard_begin(shard, vocab_offset, (Q_shard, scale_shard), ws, stream=stream, out=out)


def dg_soft_embed_shard_end_e4m3(shard: torch.Tensor, lse: torch.Tensor, Q_shard: torch.Tensor,
                                 scale_shard: torch.Tensor, gamma: float, ws: torch.Tensor,
                                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dg_soft_embed_shard_end over an 8-bit table shard (codes, row scales)."""
    return dg_soft_embed_shard_end(shard, lse, (Q_shard, scale_shard), gamma, ws, out=out, stream=stream)


def dg_row_stats_combine(states: torch.Tensor, stream=None, out: dict | None = None) -> dict:
    """Full-row statistics from [T, R, 4] shard summaries in shard order."""
    T, R = states.shape[0], states.shape[1]
    dev = states.device
    o = out if out is not None else {"m": _new(R, torch.float32, dev), "lse": _new(R, torch.float32, dev),
                                     "H": _new(R, torch.float32, dev), "kappa": _new(R, torch.float32, dev),
                                     "argmax": _new(R, torch.int32, dev)}
    _check(lib.dg_row_stats_combine(_ptr(states), T, R, _ptr(o.get("m")), _ptr(o.get("lse")), _ptr(o.get("H")),
                                    _ptr(o.get("kappa")), _ptr(o.get("argmax")), _stream(stream)),
           "dg_row_stats_combine")
    return o


def dg_row_stats_sample(logits: torch.Tensor, temperature: float = 1.0, seed: int = 0, offset: int = 0,
                        V: int | None = None, stream=None, out: dict | None = None) -> dict:
    """Row statistics and a drawn candidate in one pass; kappa = -ln p(candidate)."""
    R = logits.shape[0]
    V = logits.shape[1] if V is None else V
    dev = logits.device
    o = out if out is not None else {
        "m": _new(R, torch.float32, dev), "lse": _new(R, torch.float32, dev), "H": _new(R, torch.float32, dev),
        "kappa": _new(R, torch.float32, dev), "argmax": _new(R, torch.int32, dev),
        "candidate": _new(R, torch.int32, dev), "log_p": _new(R, torch.float32, dev)}
    _check(lib.dg_row_stats_sample(_ptr(logits), R, V, _ld(logits), temperature, seed, offset, _ptr(o.get("m")),
                                   _ptr(o.get("lse")), _ptr(o.get("H")), _ptr(o.get("kappa")),
                                   _ptr(o.get("argmax")), _ptr(o["candidate"]), _ptr(o.get("log_p")),
                                   _stream(stream)), "dg_row_stats_sample")
    return o


def dg_soft_embed_workspace_size(R: int, vocab_len: int, d: int) -> int:
    return int(lib.dg_soft_embed_workspace_size(R, vocab_len, d))


def workspace(R: int, vocab_len: int, d: int, device) -> torch.Tensor:
    """A workspace tensor large enough for dg_soft_embed / dg_sampler_step."""
    n = max(16, dg_soft_embed_workspace_size(R, vocab_len, d))
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def dg_soft_embed(logits: torch.Tensor, lse: torch.Tensor, vocab_start: int, vocab_end: int,
                  W_shard: torch.Tensor, gamma: float, out: torch.Tensor | None = None,
                  ws: torch.Tensor | None = None, stream=None, R: int | None = None) -> torch.Tensor:
    """E = gamma * softmax(logits)[:, s:e] @ W_shard[0:e-s] (W_shard: bf16 [rows_pad, >=d])."""
    R = logits.shape[0] if R is None else R
    d = W_shard.shape[1]
    if W_shard.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("W_shard must hold bfloat16 values")
    if out is None:
        out = _new((R, d), torch.float32, logits.device)
    if ws is None:
        ws = workspace(R, max(1, vocab_end - vocab_start), d, logits.device)
    _check(lib.dg_soft_embed(_ptr(logits), _ld(logits), _ptr(lse), R, vocab_start, vocab_end, _ptr(W_shard),
                             W_shard.shape[0], _ld(W_shard), d, gamma, _ptr(out), _ld(out), _ptr(ws), ws.numel(),
                             _stream(stream)), "dg_soft_embed")
    return out


def dg_soft_embed_no_alloc(logits: torch.Tensor, lse: torch.Tensor, vocab_start: int, vocab_end: int,
                           W_shard: torch.Tensor, gamma: float, out: torch.Tensor, stream=None,
                           R: int | None = None) -> torch.Tensor:
    """dg_soft_embed without a workspace: the library's fixed scratch array holds the
    partial tiles.  `out` [R, >=d] fp32 must be given; nothing is allocated."""
    R = logits.shape[0] if R is None else R
    d = W_shard.shape[1]
    _check(lib.dg_soft_embed_no_alloc(_ptr(logits), _ld(logits), _ptr(lse), R, vocab_start, vocab_end,
                                      _ptr(W_shard), W_shard.shape[0], _ld(W_shard), d, gamma, _ptr(out), _ld(out),
                                      _stream(stream)), "dg_soft_embed_no_alloc")
    return out


def dg_quantize_e4m3(W: torch.Tensor, stream=None) -> tuple:
    """Per-row E4M3 quantisation of a bf16 table [V, >=d] -> (Q, scale): Q a uint8 [V, d] view
    of a buffer whose rows are padded to a multiple of 16 bytes, scale fp32 [V]."""
    if W.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("W must hold bfloat16 values")
    V, d = W.shape
    ldq = (d + 15) // 16 * 16
    Q = _new((V, ldq), torch.uint8, W.device)
    scale = _new(V, torch.float32, W.device)
    _check(lib.dg_quantize_e4m3(_ptr(W), V, d, _ld(W), _ptr(Q), ldq, _ptr(scale), _stream(stream)),
           "dg_quantize_e4m3")
    return Q[:, :d], scale


def dg_soft_embed_workspace_size_e4m3(R: int, vocab_len: int, d: int) -> int:
    return int(lib.dg_soft_embed_workspace_size_e4m3(R, vocab_len, d))


def workspace_e4m3(R: int, vocab_len: int, d: int, device) -> torch.Tensor:
    """A workspace tensor large enough for dg_soft_embed_e4m3 / dg_sampler_step_e4m3."""
    n = max(16, dg_soft_embed_workspace_size_e4m3(R, vocab_len, d))
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def dg_soft_embed_e4m3(logits: torch.Tensor, lse: torch.Tensor, vocab_start: int, vocab_end: int,
                       Q_shard: torch.Tensor, scale_shard: torch.Tensor, gamma: float, out: torch.Tensor | None = None,
                       ws: torch.Tensor | None = None, stream=None, R: int | None = None) -> torch.Tensor:
    """E = gamma * softmax(logits)[:, s:e] @ (scale * e4m3(Q_shard))[0:e-s] (Q_shard uint8 [rows_pad, d])."""
    R = logits.shape[0] if R is None else R
    d = Q_shard.shape[1]
    if Q_shard.dtype != torch.uint8 or scale_shard.dtype != torch.float32:
        raise TypeError("Q_shard must be uint8 codes and scale_shard fp32")
    if out is None:
        out = _new((R, d), torch.float32, logits.device)
    if ws is None:
        ws = workspace_e4m3(R, max(1, vocab_end - vocab_start), d, logits.device)
    _check(lib.dg_soft_embed_e4m3(_ptr(logits), _ld(logits), _ptr(lse), R, vocab_start, vocab_end, _ptr(Q_shard),
                                  _ptr(scale_shard), Q_shard.shape[0], _ld(Q_shard), d, gamma, _ptr(out), _ld(out),
                                  _ptr(ws), ws.numel(), _stream(stream)), "dg_soft_embed_e4m3")
    return out


def dg_sampler_step_e4m3(logits: torch.Tensor, n_req: int, L_c: int, Q: torch.Tensor, scale: torch.Tensor,
                         gamma: float, budgets: torch.Tensor, min_accept: int = 0, vocab_start: int = 0,
                         vocab_end: int | None = None, V: int | None = None, out: dict | None = None,
                         ws: torch.Tensor | None = None, stream=None, two_pass: bool = False) -> dict:
    """dg_sampler_step with the 8-bit table (Q uint8 [rows_pad, d], scale fp32 [rows_pad])."""
    R = n_req * L_c
    V = logits.shape[1] if V is None else V
    vocab_end = V if vocab_end is None else vocab_end
    d = Q.shape[1]
    dev = logits.device
    o = out
    if o is None:
        o = {k: _new(R, torch.float32, dev) for k in ("m", "lse", "H", "kappa")}
        o.update(argmax=_new(R, torch.int32, dev), order=_new(R, torch.int32, dev), mask=_new(R, torch.uint8, dev),
                 n_accepted=_new(n_req, torch.int32, dev), E=_new((R, d), torch.float32, dev))
    if ws is None:
        ws = workspace_e4m3(R, max(1, vocab_end - vocab_start), d, dev)
    _check(lib.dg_sampler_step_e4m3(_ptr(logits), n_req, L_c, V, _ld(logits), _ptr(Q), _ptr(scale), vocab_start,
                                    vocab_end, Q.shape[0], _ld(Q), d, gamma, _ptr(budgets), min_accept,
                                    _ptr(o["m"]), _ptr(o["lse"]), _ptr(o["H"]), _ptr(o["kappa"]), _ptr(o["argmax"]),
                                    _ptr(o["order"]), _ptr(o["mask"]), _ptr(o["n_accepted"]), _ptr(o["E"]),
                                    _ld(o["E"]), _flags(two_pass), _ptr(ws), ws.numel(), _stream(stream)),
           "dg_sampler_step_e4m3")
    return o


def dg_entropy_accept(H: torch.Tensor, kappa: torch.Tensor, n_req: int, L_c: int, budgets: torch.Tensor,
                      min_accept: int = 0, stream=None, out: dict | None = None) -> dict:
    dev = H.device
    R = n_req * L_c
    o = out if out is not None else {"order": _new(R, torch.int32, dev), "mask": _new(R, torch.uint8, dev),
                                     "n_accepted": _new(n_req, torch.int32, dev)}
    _check(lib.dg_entropy_accept(_ptr(H), _ptr(kappa), n_req, L_c, _ptr(budgets), min_accept, _ptr(o["order"]),
                                 _ptr(o["mask"]), _ptr(o["n_accepted"]), _stream(stream)), "dg_entropy_accept")
    return o


def dg_sum_partials(partials: list, gamma: float, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    R, d = partials[0].shape
    ldp = _ld(partials[0])
    if any(tuple(p.shape) != (R, d) or _ld(p) != ldp for p in partials):
        raise ValueError("partials must share shape and leading dimension")
    if out is None:
        out = _new((R, d), torch.float32, partials[0].device)
    arr = (_p * len(partials))(*[p.data_ptr() for p in partials])
    _check(lib.dg_sum_partials(arr, len(partials), R, d, ldp, gamma, _ptr(out), _ld(out), _stream(stream)),
           "dg_sum_partials")
    return out


def dg_sampler_step(logits: torch.Tensor, n_req: int, L_c: int, W: torch.Tensor, gamma: float,
                    budgets: torch.Tensor, min_accept: int = 0, vocab_start: int = 0, vocab_end: int | None = None,
                    V: int | None = None, out: dict | None = None, ws: torch.Tensor | None = None,
                    stream=None, two_pass: bool = False) -> dict:
    """One fused sampler step; returns dict m, lse, H, kappa, argmax, order, mask, n_accepted, E.
    two_pass: statistics before the product even over the whole vocabulary (DG_STEP_TWO_PASS)."""
    R = n_req * L_c
    V = logits.shape[1] if V is None else V
    vocab_end = V if vocab_end is None else vocab_end
    d = W.shape[1]
    dev = logits.device
    o = out
    if o is None:
        o = {k: _new(R, torch.float32, dev) for k in ("m", "lse", "H", "kappa")}
        o.update(argmax=_new(R, torch.int32, dev), order=_new(R, torch.int32, dev), mask=_new(R, torch.uint8, dev),
                 n_accepted=_new(n_req, torch.int32, dev), E=_new((R, d), torch.float32, dev))
    if ws is None:
        ws = workspace(R, max(1, vocab_end - vocab_start), d, dev)
    _check(lib.dg_sampler_step(_ptr(logits), n_req, L_c, V, _ld(logits), _ptr(W), vocab_start, vocab_end,
                               W.shape[0], _ld(W), d, gamma, _ptr(budgets), min_accept, _ptr(o["m"]), _ptr(o["lse"]),
                               _ptr(o["H"]), _ptr(o["kappa"]), _ptr(o["argmax"]), _ptr(o["order"]), _ptr(o["mask"]),
                               _ptr(o["n_accepted"]), _ptr(o["E"]), _ld(o["E"]), _flags(two_pass), _ptr(ws),
                               ws.numel(), _stream(stream)), "dg_sampler_step")
    return o


def dg_entropy_accept_eligible(H: torch.Tensor, kappa: torch.Tensor, eligible: torch.Tensor, n_req: int, L_c: int,
                               budgets: torch.Tensor, min_accept: int = 0, stream=None, out: dict | None = None) -> dict:
    dev = H.device
    R = n_req * L_c
    o = out if out is not None else {"order": _new(R, torch.int32, dev), "mask": _new(R, torch.uint8, dev),
                                     "n_accepted": _new(n_req, torch.int32, dev)}
    _check(lib.dg_entropy_accept_eligible(_ptr(H), _ptr(kappa), _ptr(eligible), n_req, L_c, _ptr(budgets), min_accept,
                                          _ptr(o["order"]), _ptr(o["mask"]), _ptr(o["n_accepted"]), _stream(stream)),
           "dg_entropy_accept_eligible")
    return o


LOOP_STATE_KEYS = ("canvas", "eligible", "prev_argmax", "stable", "steps", "converged")


def new_loop_state(n_req: int, L_c: int, device, canvas0: torch.Tensor | None = None) -> dict:
    """The state buffers a denoising loop starts from, as the C API documents them:
    prev_argmax -1, stable and steps 0, every position eligible, the canvas as given."""
    R = n_req * L_c
    canvas = torch.zeros(R, dtype=torch.int32, device=device) if canvas0 is None else \
        canvas0.to(device=device, dtype=torch.int32).reshape(R).clone()
    return {"canvas": canvas, "eligible": torch.ones(R, dtype=torch.uint8, device=device),
            "prev_argmax": torch.full((R,), -1, dtype=torch.int32, device=device),
            "stable": torch.zeros(n_req, dtype=torch.int32, device=device),
            "steps": torch.zeros(n_req, dtype=torch.int32, device=device),
            "converged": torch.zeros(n_req, dtype=torch.uint8, device=device)}


def dg_loop_update(candidate: torch.Tensor, H: torch.Tensor, mask: torch.Tensor, n_req: int, L_c: int,
                   state: dict, stable_steps: int, entropy_threshold: float, step_limit: int,
                   argmax: torch.Tensor | None = None, stream=None) -> dict:
    """Updates `state` (see new_loop_state) in place after one step; returns it.  The
    canvas takes `candidate`; stability is judged on `argmax` (default: the candidates)."""
    am = candidate if argmax is None else argmax
    _check(lib.dg_loop_update(_ptr(candidate), _ptr(am), _ptr(H), _ptr(mask), n_req, L_c, stable_steps,
                              entropy_threshold,
                              step_limit, *[_ptr(state[k]) for k in LOOP_STATE_KEYS], _stream(stream)),
           "dg_loop_update")
    return state


def dg_sampler_loop_step(logits: torch.Tensor, n_req: int, L_c: int, W: torch.Tensor, gamma: float,
                         budgets: torch.Tensor, state: dict, stable_steps: int, entropy_threshold: float,
                         step_limit: int, min_accept: int = 0, vocab_start: int = 0, vocab_end: int | None = None,
                         V: int | None = None, out: dict | None = None, ws: torch.Tensor | None = None,
                         temperature: float = 0.0, seed: int = 0, offset: int = 0, stream=None,
                         two_pass: bool = False) -> dict:
    """One denoising-loop step: the fused step over the eligible positions, then the loop
    update of `state` in place.  Returns the step outputs as dg_sampler_step does, plus
    `candidate` (the drawn tokens) when temperature > 0."""
    R = n_req * L_c
    V = logits.shape[1] if V is None else V
    vocab_end = V if vocab_end is None else vocab_end
    d = W.shape[1]
    dev = logits.device
    o = out
    if o is None:
        o = {k: _new(R, torch.float32, dev) for k in ("m", "lse", "H", "kappa")}
        o.update(argmax=_new(R, torch.int32, dev), order=_new(R, torch.int32, dev), mask=_new(R, torch.uint8, dev),
                 n_accepted=_new(n_req, torch.int32, dev), E=_new((R, d), torch.float32, dev))
    if temperature != 0.0 and "candidate" not in o:
        o["candidate"] = _new(R, torch.int32, dev)
    if ws is None:
        ws = workspace(R, max(1, vocab_end - vocab_start), d, dev)
    _check(lib.dg_sampler_loop_step(_ptr(logits), n_req, L_c, V, _ld(logits), _ptr(W), vocab_start, vocab_end,
                                    W.shape[0], _ld(W), d, gamma, _ptr(budgets), min_accept, stable_steps,
                                    entropy_threshold, step_limit, temperature, seed, offset, _ptr(o["m"]),
                                    _ptr(o["lse"]), _ptr(o["H"]), _ptr(o["kappa"]), _ptr(o["argmax"]),
                                    _ptr(o.get("candidate")), _ptr(o["order"]), _ptr(o["mask"]),
                                    _ptr(o["n_accepted"]), _ptr(o["E"]), _ld(o["E"]),
                                    *[_ptr(state[k]) for k in LOOP_STATE_KEYS], _flags(two_pass), _ptr(ws),
                                    ws.numel(), _stream(stream)), "dg_sampler_loop_step")
    return o


def dg_sampler_loop_step_e4m3(logits: torch.Tensor, n_req: int, L_c: int, Q: torch.Tensor, scale: torch.Tensor,
                              gamma: float, budgets: torch.Tensor, state: dict, stable_steps: int,
                              entropy_threshold: float, step_limit: int, min_accept: int = 0, vocab_start: int = 0,
                              vocab_end: int | None = None, V: int | None = None, out: dict | None = None,
                              ws: torch.Tensor | None = None, temperature: float = 0.0, seed: int = 0, offset: int = 0,
                              stream=None, two_pass: bool = False) -> dict:
    """dg_sampler_loop_step with the 8-bit table (Q uint8 [rows_pad, d], scale fp32 [rows_pad])."""
    R = n_req * L_c
    V = logits.shape[1] if V is None else V
    vocab_end = V if vocab_end is None else vocab_end
    d = Q.shape[1]
    dev = logits.device
    o = out
    if o is None:
        o = {k: _new(R, torch.float32, dev) for k in ("m", "lse", "H", "kappa")}
        o.update(argmax=_new(R, torch.int32, dev), order=_new(R, torch.int32, dev), mask=_new(R, torch.uint8, dev),
                 n_accepted=_new(n_req, torch.int32, dev), E=_new((R, d), torch.float32, dev))
    if temperature != 0.0 and "candidate" not in o:
        o["candidate"] = _new(R, torch.int32, dev)
    if ws is None:
        ws = workspace_e4m3(R, max(1, vocab_end - vocab_start), d, dev)
    _check(lib.dg_sampler_loop_step_e4m3(_ptr(logits), n_req, L_c, V, _ld(logits), _ptr(Q), _ptr(scale), vocab_start,
                                         vocab_end, Q.shape[0], _ld(Q), d, gamma, _ptr(budgets), min_accept,
                                         stable_steps, entropy_threshold, step_limit, temperature, seed, offset,
                                         _ptr(o["m"]), _ptr(o["lse"]), _ptr(o["H"]), _ptr(o["kappa"]),
                                         _ptr(o["argmax"]), _ptr(o.get("candidate")), _ptr(o["order"]),
                                         _ptr(o["mask"]), _ptr(o["n_accepted"]), _ptr(o["E"]), _ld(o["E"]),
                                         *[_ptr(state[k]) for k in LOOP_STATE_KEYS], _flags(two_pass), _ptr(ws),
                                         ws.numel(), _stream(stream)), "dg_sampler_loop_step_e4m3")
    return o


def dg_get_device_status(stream=None) -> None:
    _check(lib.dg_get_device_status(_stream(stream)), "dg_get_device_status")


def dg_check_wait_timeout(limit_us: int, stream=None) -> None:
    """Queues the diagnostic wait that gives up after limit_us; the next
    dg_get_device_status() raises DgError with DG_ERR_TIMEOUT."""
    _check(lib.dg_check_wait_timeout(int(limit_us), _stream(stream)), "dg_check_wait_timeout")
