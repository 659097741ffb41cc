"""Python binding of the DSpark draft-sampling / verification library (sm_103a).

Thin argument marshalling over the C ABI of ``include/dspark.h``: each
function below has the name of the C entry point it calls, takes torch CUDA
tensors, passes their device pointers, sizes and the current CUDA stream, and
raises ``DSparkError`` on a non-OK status.  Every step of the computation runs
in the library's CUDA kernels; there is no fallback of any kind -- if
``libdspark.so`` has not been built, importing a function fails loudly.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "DSparkError", "lib", "Workspace", "OP_DRAFT_LOGITS", "OP_MARKOV_SAMPLE", "OP_VERIFY",
    "OP_SCHEDULE", "OP_VERIFY_GREEDY", "OP_CONFIDENCE", "OP_VERIFY_LOGITS", "OP_VERIFY_GUMBEL",
    "dspark_workspace_size", "dspark_verify_gumbel",
    "dspark_verify_greedy", "dspark_verify_logits",
    "dspark_confidence", "dspark_markov_sample_reduced", "dspark_markov_sample_conf", "D2T_INDEX", "D2T_OFFSET", "dspark_draft_logits", "dspark_markov_sample",
    "dspark_verify", "dspark_schedule", "dspark_read_status", "dspark_status_string",
    "dspark_selftest_wait_timeout", "STATUS_TIMEOUT", "STATUS_NUMERIC", "STATUS_INPUT_RANGE",
    "STATUS_INTERNAL", "STATUS_INDEX",
]

# The library this binding loads: the in-tree build, or the file DSPARK_LIBRARY names (another
# build of the same sources, e.g. one compiled with -DDSPARK_CHECKED).
LIB_PATH = os.environ.get("DSPARK_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdspark.so")

OP_DRAFT_LOGITS, OP_MARKOV_SAMPLE, OP_VERIFY, OP_SCHEDULE, OP_VERIFY_GREEDY, OP_CONFIDENCE = 0, 1, 2, 3, 4, 5
OP_VERIFY_LOGITS = 6
OP_VERIFY_GUMBEL = 7
F32, BF16 = 0, 1
D2T_INDEX, D2T_OFFSET = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NUMERIC, ERR_INPUT_RANGE = range(7)
STATUS_TIMEOUT, STATUS_NUMERIC, STATUS_INPUT_RANGE, STATUS_INTERNAL, STATUS_INDEX = 0x1, 0x2, 0x4, 0x8, 0x10

_lib = None


class DSparkError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(the DSpark ops exist only as CUDA kernels)")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u64, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p
    L.dspark_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.dspark_workspace_size.restype = sz
    L.dspark_draft_logits.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, sz, vp]
    L.dspark_markov_sample.argtypes = [vp, vp, vp, vp, i32, vp, u64, u64, i32, i32, i32, i32,
                                       vp, vp, vp, sz, vp]
    L.dspark_markov_sample_conf.argtypes = [vp, vp, vp, vp, i32, vp, u64, u64, i32, i32, i32, i32,
                                            vp, i32, i32, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_markov_sample_reduced.argtypes = [vp, vp, vp, vp, i32, vp, u64, u64, i32, i32, i32, i32,
                                               vp, i32, i32, vp, vp, vp, sz, vp]
    L.dspark_verify.argtypes = [vp, vp, vp, vp, u64, u64, i32, i32, i32, vp, vp, vp, sz, vp]
    L.dspark_verify_greedy.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.dspark_verify_gumbel.argtypes = [vp, vp, vp, vp, u64, u64, i32, i32, i32, vp, vp, vp, sz, vp]
    L.dspark_verify_logits.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, u64, u64, i32, i32, i32,
                                       vp, vp, vp, sz, vp]
    L.dspark_confidence.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, ctypes.c_float, vp, i32, i32, i32, i32, i32,
                                    vp, vp, sz, vp]
    L.dspark_schedule.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_read_status.argtypes = [vp, u32p, vp]
    L.dspark_status_string.argtypes = [i32]
    L.dspark_status_string.restype = ctypes.c_char_p
    L.dspark_last_error.argtypes = []
    L.dspark_last_error.restype = ctypes.c_char_p
    L.dspark_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_longlong, vp]
    for f in ("dspark_draft_logits", "dspark_markov_sample", "dspark_verify", "dspark_schedule",
              "dspark_read_status", "dspark_selftest_wait_timeout"):
        getattr(L, f).restype = i32
    _lib = L
    return L


def _check(status: int, where: str):
    if status != OK:
        msg = lib().dspark_last_error().decode() or lib().dspark_status_string(status).decode()
        raise DSparkError(status, where, msg)


def _torch():
    import torch
    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t):
    """Library dtype code of a bf16 or fp32 tensor."""
    return BF16 if t.dtype == _torch().bfloat16 else F32


def _need(t, name, dtypes, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")


def dspark_workspace_size(op: int, B: int = 0, N: int = 0, V: int = 0, r: int = 0) -> int:
    return int(lib().dspark_workspace_size(op, B, N, V, r))


class Workspace:
    """Device workspace for one op (256-byte aligned torch allocation, reused across calls)."""

    def __init__(self, op: int, B: int = 0, N: int = 0, V: int = 0, r: int = 0, device=None):
        torch = _torch()
        self.nbytes = dspark_workspace_size(op, B, N, V, r)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8,
                               device=device if device is not None else "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.view = self.buf[off:off + self.nbytes]

    @property
    def ptr(self):
        return ctypes.c_void_p(self.view.data_ptr())


def _ws(ws, op, B=0, N=0, V=0, r=0, device=None):
    return ws if ws is not None else Workspace(op, B, N, V, r, device)


def dspark_draft_logits(hidden, lm_head, logits=None, workspace=None, stream=None):
    """logits[m, v] = sum_h hidden[m, h] * lm_head[v, h]  (hidden [M,H], lm_head [V,H]; bf16 or fp32)."""
    torch = _torch()
    _need(hidden, "hidden", (torch.bfloat16, torch.float32), 2)
    _need(lm_head, "lm_head", (hidden.dtype,), 2)
    M, H = hidden.shape
    V = lm_head.shape[0]
    if lm_head.shape[1] != H:
        raise ValueError("lm_head must be [V, H] with the hidden size of `hidden`")
    if logits is None:
        logits = torch.empty(M, V, dtype=torch.float32, device=hidden.device)
    _need(logits, "logits", (torch.float32,))
    ws = _ws(workspace, OP_DRAFT_LOGITS, device=hidden.device)
    dt = BF16 if hidden.dtype == torch.bfloat16 else F32
    _check(lib().dspark_draft_logits(_ptr(hidden), _ptr(lm_head), dt, M, H, V, _ptr(logits),
                                     ws.ptr, ws.nbytes, _stream(stream)), "dspark_draft_logits")
    return logits


def dspark_markov_sample(base_logits, anchor, w1, w2, temperature, seed: int, offset: int,
                         draft_tokens=None, lse=None, workspace=None, stream=None):
    """Sequential Markov-biased Gumbel-max sampling; returns draft_tokens [B, N] int32.

    base_logits [B, N, V] fp32, anchor [B] int32, w1/w2 [V, r] (bf16 or fp32),
    temperature [B] fp32.  Pass an fp32 [B, N] tensor as `lse` to receive the
    log-sum-exp of each step's scaled logits.
    """
    torch = _torch()
    _need(base_logits, "base_logits", (torch.float32,), 3)
    _need(anchor, "anchor", (torch.int32,), 1)
    _need(w1, "w1", (torch.bfloat16, torch.float32), 2)
    _need(w2, "w2", (w1.dtype,), 2)
    _need(temperature, "temperature", (torch.float32,), 1)
    B, N, V = base_logits.shape
    r = w1.shape[1]
    if tuple(w2.shape) != (V, r) or w1.shape[0] != V:
        raise ValueError("w1 and w2 must both be [V, r]")
    if draft_tokens is None:
        draft_tokens = torch.empty(B, N, dtype=torch.int32, device=base_logits.device)
    _need(draft_tokens, "draft_tokens", (torch.int32,))
    if lse is not None:
        _need(lse, "lse", (torch.float32,))
    ws = _ws(workspace, OP_MARKOV_SAMPLE, B, N, V, r, base_logits.device)
    dt = BF16 if w1.dtype == torch.bfloat16 else F32
    _check(lib().dspark_markov_sample(_ptr(base_logits), _ptr(anchor), _ptr(w1), _ptr(w2), dt,
                                      _ptr(temperature), seed, offset, B, N, V, r,
                                      _ptr(draft_tokens), _ptr(lse), ws.ptr, ws.nbytes,
                                      _stream(stream)), "dspark_markov_sample")
    return draft_tokens


def dspark_markov_sample_conf(base_logits, anchor, w1, w2, temperature, seed: int, offset: int, hidden, w_h, w_e,
                              beta: float, tau, draft_tokens=None, conf=None, lse=None, workspace=None, stream=None):
    """dspark_markov_sample with the calibrated confidence head evaluated at every step; returns
    (draft_tokens [B, N] int32, conf [B, N] fp32).  hidden [B*N, H] (bf16 or fp32), w_h [H], w_e [r],
    tau [N] fp32; conf[b, i] is the conditional acceptance probability of draft token (b, i)."""
    torch = _torch()
    _need(base_logits, "base_logits", (torch.float32,), 3)
    _need(anchor, "anchor", (torch.int32,), 1)
    _need(w1, "w1", (torch.bfloat16, torch.float32), 2)
    _need(w2, "w2", (w1.dtype,), 2)
    _need(temperature, "temperature", (torch.float32,), 1)
    _need(hidden, "hidden", (torch.bfloat16, torch.float32), 2)
    _need(w_h, "w_h", (torch.float32,), 1)
    _need(w_e, "w_e", (torch.float32,), 1)
    _need(tau, "tau", (torch.float32,), 1)
    B, N, V = base_logits.shape
    r = w1.shape[1]
    H = hidden.shape[1]
    if tuple(w2.shape) != (V, r) or w1.shape[0] != V:
        raise ValueError("w1 and w2 must both be [V, r]")
    if hidden.shape[0] != B * N or w_h.shape[0] != H or w_e.shape[0] != r or tau.shape[0] != N:
        raise ValueError("shapes: hidden [B*N, H], w_h [H], w_e [r], tau [N]")
    if draft_tokens is None:
        draft_tokens = torch.empty(B, N, dtype=torch.int32, device=base_logits.device)
    if conf is None:
        conf = torch.empty(B, N, dtype=torch.float32, device=base_logits.device)
    _need(draft_tokens, "draft_tokens", (torch.int32,))
    _need(conf, "conf", (torch.float32,))
    if lse is not None:
        _need(lse, "lse", (torch.float32,))
    ws = _ws(workspace, OP_MARKOV_SAMPLE, B, N, V, r, base_logits.device)
    _check(lib().dspark_markov_sample_conf(_ptr(base_logits), _ptr(anchor), _ptr(w1), _ptr(w2), _dt(w1),
                                           _ptr(temperature), seed, offset, B, N, V, r, _ptr(hidden), _dt(hidden), H,
                                           _ptr(w_h), _ptr(w_e), float(beta), _ptr(tau), _ptr(draft_tokens),
                                           _ptr(conf), _ptr(lse), ws.ptr, ws.nbytes, _stream(stream)),
           "dspark_markov_sample_conf")
    return draft_tokens, conf


def dspark_markov_sample_reduced(base_logits, anchor, w1, w2, temperature, seed: int, offset: int, d2t,
                                 mode: int, V_target: int, draft_tokens=None, lse=None, workspace=None,
                                 stream=None):
    """dspark_markov_sample on a reduced draft vocabulary (V = base_logits.shape[2]); the tokens come
    back as target-vocabulary ids through `d2t` [V] int32 (mode D2T_INDEX: d2t[d]; D2T_OFFSET:
    d + d2t[d])."""
    torch = _torch()
    _need(base_logits, "base_logits", (torch.float32,), 3)
    _need(anchor, "anchor", (torch.int32,), 1)
    _need(w1, "w1", (torch.bfloat16, torch.float32), 2)
    _need(w2, "w2", (w1.dtype,), 2)
    _need(temperature, "temperature", (torch.float32,), 1)
    _need(d2t, "d2t", (torch.int32,), 1)
    B, N, V = base_logits.shape
    r = w1.shape[1]
    if tuple(w2.shape) != (V, r) or w1.shape[0] != V or d2t.shape[0] != V:
        raise ValueError("w1 and w2 must both be [V, r] and d2t [V] over the draft vocabulary")
    if draft_tokens is None:
        draft_tokens = torch.empty(B, N, dtype=torch.int32, device=base_logits.device)
    ws = _ws(workspace, OP_MARKOV_SAMPLE, B, N, V, r, base_logits.device)
    _check(lib().dspark_markov_sample_reduced(_ptr(base_logits), _ptr(anchor), _ptr(w1), _ptr(w2), _dt(w1),
                                              _ptr(temperature), seed, offset, B, N, V, r, _ptr(d2t), int(mode),
                                              int(V_target), _ptr(draft_tokens), _ptr(lse), ws.ptr, ws.nbytes,
                                              _stream(stream)), "dspark_markov_sample_reduced")
    return draft_tokens


def dspark_verify(p_target, p_draft, draft_tokens, lengths, seed: int, offset: int,
                  out_tokens=None, num_accepted=None, workspace=None, stream=None):
    """Lossless rejection-sampling verification; returns (out_tokens [B, gamma+1], num_accepted [B])."""
    torch = _torch()
    _need(p_target, "p_target", (torch.float32,), 3)
    _need(p_draft, "p_draft", (torch.float32,), 3)
    _need(draft_tokens, "draft_tokens", (torch.int32,), 2)
    B, gamma, V = p_draft.shape
    if tuple(p_target.shape) != (B, gamma + 1, V) or tuple(draft_tokens.shape) != (B, gamma):
        raise ValueError("shapes must be p_target [B, gamma+1, V], p_draft [B, gamma, V], tokens [B, gamma]")
    if lengths is not None:
        _need(lengths, "lengths", (torch.int32,), 1)
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=p_target.device)
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=p_target.device)
    ws = _ws(workspace, OP_VERIFY, B, gamma, V, 0, p_target.device)
    _check(lib().dspark_verify(_ptr(p_target), _ptr(p_draft), _ptr(draft_tokens), _ptr(lengths),
                               seed, offset, B, gamma, V, _ptr(out_tokens), _ptr(num_accepted),
                               ws.ptr, ws.nbytes, _stream(stream)), "dspark_verify")
    return out_tokens, num_accepted


def dspark_verify_gumbel(target_logits, temperature, draft_tokens, lengths, seed: int, offset: int,
                         out_tokens=None, num_accepted=None, workspace=None, stream=None):
    """Verification with the draft's Gumbel noise (the draft sampler's seed and offset); returns
    (out_tokens [B, gamma+1], num_accepted [B])."""
    torch = _torch()
    _need(target_logits, "target_logits", (torch.float32,), 3)
    _need(temperature, "temperature", (torch.float32,), 1)
    _need(draft_tokens, "draft_tokens", (torch.int32,), 2)
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if tuple(draft_tokens.shape) != (B, gamma) or temperature.shape[0] != B:
        raise ValueError("shapes must be target_logits [B, gamma+1, V], temperature [B], tokens [B, gamma]")
    if lengths is not None:
        _need(lengths, "lengths", (torch.int32,), 1)
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=target_logits.device)
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    ws = _ws(workspace, OP_VERIFY_GUMBEL, B, gamma, 0, 0, target_logits.device)
    _check(lib().dspark_verify_gumbel(_ptr(target_logits), _ptr(temperature), _ptr(draft_tokens), _ptr(lengths),
                                      seed, offset, B, gamma, V, _ptr(out_tokens), _ptr(num_accepted), ws.ptr,
                                      ws.nbytes, _stream(stream)),
           "dspark_verify_gumbel")
    return out_tokens, num_accepted


def dspark_verify_greedy(target, draft_tokens, lengths=None, out_tokens=None, num_accepted=None,
                         workspace=None, stream=None):
    """Greedy (temperature-0) verification; returns (out_tokens [B, gamma+1], num_accepted [B])."""
    torch = _torch()
    _need(target, "target", (torch.float32,), 3)
    _need(draft_tokens, "draft_tokens", (torch.int32,), 2)
    B, g1, V = target.shape
    gamma = g1 - 1
    if tuple(draft_tokens.shape) != (B, gamma):
        raise ValueError("shapes must be target [B, gamma+1, V], tokens [B, gamma]")
    if lengths is not None:
        _need(lengths, "lengths", (torch.int32,), 1)
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=target.device)
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=target.device)
    ws = _ws(workspace, OP_VERIFY_GREEDY, B, gamma, 0, 0, target.device)
    _check(lib().dspark_verify_greedy(_ptr(target), _ptr(draft_tokens), _ptr(lengths), B, gamma, V,
                                      _ptr(out_tokens), _ptr(num_accepted), ws.ptr, ws.nbytes, _stream(stream)),
           "dspark_verify_greedy")
    return out_tokens, num_accepted


def dspark_verify_logits(target_logits, target_temperature, base_logits, anchor, w1, w2, draft_temperature,
                         draft_lse, draft_tokens, lengths, seed: int, offset: int, out_tokens=None,
                         num_accepted=None, workspace=None, stream=None):
    """Lossless verification from logits with the draft distribution recomputed;
    returns (out_tokens [B, gamma+1], num_accepted [B])."""
    torch = _torch()
    _need(target_logits, "target_logits", (torch.float32,), 3)
    _need(base_logits, "base_logits", (torch.float32,), 3)
    _need(target_temperature, "target_temperature", (torch.float32,), 1)
    _need(draft_temperature, "draft_temperature", (torch.float32,), 1)
    _need(anchor, "anchor", (torch.int32,), 1)
    _need(w1, "w1", (torch.bfloat16, torch.float32), 2)
    _need(w2, "w2", (w1.dtype,), 2)
    _need(draft_lse, "draft_lse", (torch.float32,), 2)
    _need(draft_tokens, "draft_tokens", (torch.int32,), 2)
    B, gamma, V = base_logits.shape
    r = w1.shape[1]
    if (tuple(target_logits.shape) != (B, gamma + 1, V) or tuple(draft_tokens.shape) != (B, gamma)
            or tuple(draft_lse.shape) != (B, gamma) or tuple(w1.shape) != (V, r) or tuple(w2.shape) != (V, r)
            or anchor.shape[0] != B or target_temperature.shape[0] != B or draft_temperature.shape[0] != B):
        raise ValueError("shapes: target_logits [B, gamma+1, V], base_logits [B, gamma, V], w1/w2 [V, r], "
                         "draft_lse / draft_tokens [B, gamma], anchor / temperatures [B]")
    if lengths is not None:
        _need(lengths, "lengths", (torch.int32,), 1)
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=target_logits.device)
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    ws = _ws(workspace, OP_VERIFY_LOGITS, B, gamma, V, r, target_logits.device)
    _check(lib().dspark_verify_logits(_ptr(target_logits), _ptr(target_temperature), _ptr(base_logits),
                                      _ptr(anchor), _ptr(w1), _ptr(w2), _dt(w1), r, _ptr(draft_temperature),
                                      _ptr(draft_lse), _ptr(draft_tokens), _ptr(lengths), seed, offset, B, gamma,
                                      V, _ptr(out_tokens), _ptr(num_accepted), ws.ptr, ws.nbytes,
                                      _stream(stream)), "dspark_verify_logits")
    return out_tokens, num_accepted


def dspark_confidence(hidden, w1, anchor, draft_tokens, w_h, w_e, beta: float, tau, conf=None,
                      workspace=None, stream=None):
    """Calibrated confidence head; returns conf [B, N] (the scheduler's cond_accept)."""
    torch = _torch()
    _need(hidden, "hidden", (torch.bfloat16, torch.float32), 2)
    _need(w1, "w1", (torch.bfloat16, torch.float32), 2)
    _need(anchor, "anchor", (torch.int32,), 1)
    _need(draft_tokens, "draft_tokens", (torch.int32,), 2)
    _need(w_h, "w_h", (torch.float32,), 1)
    _need(w_e, "w_e", (torch.float32,), 1)
    _need(tau, "tau", (torch.float32,), 1)
    B, N = draft_tokens.shape
    H = hidden.shape[1]
    V, r = w1.shape
    if hidden.shape[0] != B * N or anchor.shape[0] != B or w_h.shape[0] != H or w_e.shape[0] != r \
            or tau.shape[0] != N:
        raise ValueError("shapes: hidden [B*N, H], w1 [V, r], anchor [B], tokens [B, N], w_h [H], w_e [r], tau [N]")
    if conf is None:
        conf = torch.empty(B, N, dtype=torch.float32, device=hidden.device)
    ws = _ws(workspace, OP_CONFIDENCE, B, N, V, r, hidden.device)
    _check(lib().dspark_confidence(_ptr(hidden), _dt(hidden), _ptr(w1), _dt(w1), _ptr(anchor), _ptr(draft_tokens),
                                   _ptr(w_h), _ptr(w_e), float(beta), _ptr(tau), B, N, H, V, r, _ptr(conf),
                                   ws.ptr, ws.nbytes, _stream(stream)), "dspark_confidence")
    return conf


def dspark_schedule(cond_accept, sps, K_in: int, survival=None, K_out=None, lengths=None,
                    selected=None, workspace=None, stream=None):
    """Confidence-scheduled admission; returns (survival, K_out [1], lengths [B], selected [B*N])."""
    torch = _torch()
    _need(cond_accept, "cond_accept", (torch.float32,), 2)
    B, N = cond_accept.shape
    dev = cond_accept.device
    S = 0
    if sps is not None:
        _need(sps, "sps", (torch.float64,), 1)
        S = sps.shape[0]
    survival = torch.empty(B, N, dtype=torch.float32, device=dev) if survival is None else survival
    K_out = torch.empty(1, dtype=torch.int32, device=dev) if K_out is None else K_out
    lengths = torch.empty(B, dtype=torch.int32, device=dev) if lengths is None else lengths
    selected = torch.empty(B * N, dtype=torch.int32, device=dev) if selected is None else selected
    ws = _ws(workspace, OP_SCHEDULE, B, N, device=dev)
    _check(lib().dspark_schedule(_ptr(cond_accept), _ptr(sps), S, B, N, K_in, _ptr(survival),
                                 _ptr(K_out), _ptr(lengths), _ptr(selected), ws.ptr, ws.nbytes,
                                 _stream(stream)), "dspark_schedule")
    return survival, K_out, lengths, selected


def dspark_read_status(workspace: Workspace, stream=None):
    """(status code, raw status bits) of the last call that used `workspace` (synchronises)."""
    bits = ctypes.c_uint32(0)
    st = lib().dspark_read_status(workspace.ptr, ctypes.byref(bits), _stream(stream))
    if st == ERR_CUDA:
        _check(st, "dspark_read_status")
    return int(st), int(bits.value)


def dspark_status_string(status: int) -> str:
    return lib().dspark_status_string(status).decode()


def dspark_selftest_wait_timeout(workspace: Workspace, timeout_ns: int, stream=None):
    _check(lib().dspark_selftest_wait_timeout(workspace.ptr, workspace.nbytes, int(timeout_ns),
                                              _stream(stream)), "dspark_selftest_wait_timeout")
