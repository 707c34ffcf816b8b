"""Thin ctypes binding over ``librlcs.so`` (the C ABI in include/rlcs.h).

Argument marshalling only: every step of every estimator runs in the CUDA
library. PyTorch supplies device memory (inputs, outputs, workspace) and the
current CUDA stream. The functions carry the C ABI's names and raise
``RlcsError`` on any non-OK status. There is no CPU fallback: if the library
is missing, importing this module raises.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlcs.so")

RLCS_OK = 0
RLCS_SHAPE_AUTO, RLCS_SHAPE_WARP_ROW, RLCS_SHAPE_BLOCK_CHUNK, RLCS_SHAPE_BLOCK_TILE = 0, 1, 2, 3


class RlcsError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.rlcs_status_string(status).decode()
        super().__init__("%s: %s (status %d)" % (where, msg, status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "librlcs.so is not built (%s); run linear_recurrence_scan_affine_gb300.build.build()"
            % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    # F: the scalars (gamma, lambda, rho_bar, c_bar) travel as double
    P, I64, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
    sig = {
        "rlcs_workspace_bytes": ([I64, I64], SZ),
        "rlcs_workspace_bytes_tm": ([I64, I64], SZ),
        "rlcs_workspace_init": ([P, SZ, P], ctypes.c_int),
        "rlcs_check_status": ([P, P], ctypes.c_int),
        "rlcs_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "rlcs_set_shape_override": ([ctypes.c_int, I64], ctypes.c_int),
        "rlcs_gae": ([P] * 7 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_lambda_returns": ([P] * 7 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_discounted_returns": ([P] * 6 + [I64, I64, F, P, SZ, P], ctypes.c_int),
        "rlcs_vtrace": ([P] * 9 + [I64, I64, F, F, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_retrace": ([P] * 9 + [I64, I64, F, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_eligibility_traces": ([P] * 3 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_episodic_prefix_sum": ([P] * 3 + [I64, I64, P, SZ, P], ctypes.c_int),
        "rlcs_gae_and_returns": ([P] * 8 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_affine_scan": ([P] * 5 + [I64, I64, ctypes.c_int, P, SZ, P], ctypes.c_int),
        "rlcs_gae_compact": ([P] * 7 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_diag_stream_copy": ([P, ctypes.c_int, P, I64, I64, ctypes.c_int, P], ctypes.c_int),
        "rlcs_gae_tm": ([P] * 7 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_lambda_returns_tm": ([P] * 7 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_discounted_returns_tm": ([P] * 6 + [I64, I64, F, P, SZ, P], ctypes.c_int),
        "rlcs_vtrace_tm": ([P] * 9 + [I64, I64, F, F, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_retrace_tm": ([P] * 9 + [I64, I64, F, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_eligibility_traces_tm": ([P] * 3 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_episodic_prefix_sum_tm": ([P] * 3 + [I64, I64, P, SZ, P], ctypes.c_int),
        "rlcs_gae_and_returns_tm": ([P] * 8 + [I64, I64, F, F, P, SZ, P], ctypes.c_int),
        "rlcs_run_group": ([P, ctypes.c_int, P, SZ, P], ctypes.c_int),
        "rlcs_group_workspace_bytes": ([P, ctypes.c_int], SZ),
        "rlcs_affine_scan_tm": ([P] * 5 + [I64, I64, ctypes.c_int, P, SZ, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()
EXPORTED = ("rlcs_workspace_bytes", "rlcs_workspace_init", "rlcs_check_status",
            "rlcs_status_string", "rlcs_set_shape_override", "rlcs_gae",
            "rlcs_lambda_returns", "rlcs_discounted_returns", "rlcs_vtrace",
            "rlcs_retrace", "rlcs_eligibility_traces", "rlcs_episodic_prefix_sum",
            "rlcs_gae_and_returns", "rlcs_affine_scan", "rlcs_gae_compact",
            "rlcs_diag_stream_copy", "rlcs_workspace_bytes_tm", "rlcs_gae_tm",
            "rlcs_lambda_returns_tm",
            "rlcs_discounted_returns_tm", "rlcs_vtrace_tm", "rlcs_retrace_tm",
            "rlcs_eligibility_traces_tm", "rlcs_episodic_prefix_sum_tm",
            "rlcs_gae_and_returns_tm", "rlcs_affine_scan_tm", "rlcs_run_group",
            "rlcs_group_workspace_bytes")


def lib():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def _check(status, where):
    if status != RLCS_OK:
        raise RlcsError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# One zeroed workspace per (device, stream), grown on demand. A workspace is
# reused only by calls on its own stream, which the stream orders.
_ws_lock = threading.Lock()
_ws_cache = {}


def workspace_for(N, T, device, stream=None, need=None):
    """The cached workspace of (device, stream), grown to `need` bytes (default:
    what a row-major [N, T] call needs)."""
    if need is None:
        need = _lib.rlcs_workspace_bytes(N, T)
    if need == 0:
        return None, 0
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           s.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            # zeroed on the stream that will use it, so the fill is ordered
            # before the first call (and the memory belongs to that stream)
            with torch.cuda.stream(s):
                ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws, ws.numel()


def _rows(t, name, dtype=torch.float32):
    if t.dim() == 1:
        t = t.unsqueeze(0)
    if t.dim() != 2:
        raise ValueError("%s must be [N, T] (or [T])" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.contiguous()


def _opt(t, name, N, T):
    if t is None:
        return None
    t = _rows(t, name)
    if t.shape != (N, T):
        raise ValueError("%s must have shape (%d, %d)" % (name, N, T))
    return t


def _boot(b, N):
    if b is None:
        return None
    b = b.reshape(-1)
    if not b.is_cuda or b.dtype != torch.float32 or b.numel() != N:
        raise ValueError("bootstrap_value must be a float32 CUDA tensor of %d values" % N)
    return b.contiguous()


def _prep(main, others, rewards_name="rewards"):
    r = _rows(main, rewards_name)
    N, T = r.shape
    outs = [r]
    for t, name in others:
        x = _rows(t, name)
        if x.shape != (N, T):
            raise ValueError("%s must have shape (%d, %d)" % (name, N, T))
        outs.append(x)
    return N, T, outs


def _finish(out, like):
    return out.reshape(like.shape)


def _out(t, name, like, dtype=None):
    """A caller-provided output, written in place. The library writes N*T
    elements from its first address and cannot see the buffer's size, so it
    must be a contiguous CUDA tensor on the inputs' device, with their element
    count and the output's dtype (the inputs' unless stated)."""
    dtype = like.dtype if dtype is None else dtype
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device != like.device:
        raise ValueError("%s must be on %s, got %s" % (name, like.device, t.device))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.numel() != like.numel() or not t.is_contiguous():
        raise ValueError("%s must be a contiguous tensor of %d elements" % (name, like.numel()))
    return t


def _devices(main, *tensors, stream=None):
    """Every array of a call on one CUDA device, the current one (the library
    launches there), and the stream, if one is given, on that device too."""
    dev = main.device
    for t in tensors:
        if t is not None and t.device != dev:
            raise ValueError("every array of a call must be on %s; one is on %s" % (dev, t.device))
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError("the arrays are on %s but the current CUDA device is cuda:%d; call under "
                         "torch.cuda.device(%s)" % (dev, cur, dev))
    if stream is not None and stream.device != dev:
        raise ValueError("the stream is on %s, the arrays on %s" % (stream.device, dev))


def rlcs_gae(rewards, values, terminateds, gamma=0.99, lambda_=0.95, bootstrap_value=None,
             truncateds=None, next_values=None, out=None, stream=None):
    N, T, (r, v, d) = _prep(rewards, [(values, "values"), (terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, d, tr, nv, b, o, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_gae(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b), _ptr(o),
                         N, T, gamma, lambda_, _ptr(ws), wsb, _stream(stream)), "rlcs_gae")
    return _finish(o, rewards)


def rlcs_lambda_returns(rewards, values, terminateds, gamma=0.99, lambda_=0.95,
                        bootstrap_value=None, truncateds=None, next_values=None, out=None,
                        stream=None):
    N, T, (r, v, d) = _prep(rewards, [(values, "values"), (terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, d, tr, nv, b, o, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_lambda_returns(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                                    _ptr(o), N, T, gamma, lambda_, _ptr(ws), wsb,
                                    _stream(stream)), "rlcs_lambda_returns")
    return _finish(o, rewards)


def rlcs_discounted_returns(rewards, terminateds, gamma=0.99, bootstrap_value=None,
                            truncateds=None, next_values=None, out=None, stream=None):
    N, T, (r, d) = _prep(rewards, [(terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, d, tr, nv, b, o, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_discounted_returns(_ptr(r), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b), _ptr(o),
                                        N, T, gamma, _ptr(ws), wsb, _stream(stream)),
           "rlcs_discounted_returns")
    return _finish(o, rewards)


def rlcs_vtrace(rewards, values, log_rhos, terminateds, gamma=0.99, lambda_=1.0, rho_bar=1.0,
                c_bar=1.0, bootstrap_value=None, truncateds=None, next_values=None,
                with_pg=True, out=None, out_pg=None, stream=None):
    """Returns (vs, pg_advantages); pg_advantages is None when with_pg=False."""
    N, T, (r, v, lr, d) = _prep(rewards, [(values, "values"), (log_rhos, "log_rhos"),
                                          (terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    vs = torch.empty_like(r) if out is None else _out(out, "out", r)
    pg = (torch.empty_like(r) if out_pg is None else _out(out_pg, "out_pg", r)) if with_pg else None
    _devices(r, v, lr, d, tr, nv, b, vs, pg, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_vtrace(_ptr(r), _ptr(v), _ptr(lr), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                            _ptr(vs), _ptr(pg), N, T, gamma, lambda_, rho_bar, c_bar,
                            _ptr(ws), wsb, _stream(stream)), "rlcs_vtrace")
    return _finish(vs, rewards), (None if pg is None else _finish(pg, rewards))


def rlcs_retrace(rewards, values, q_values, log_rhos, terminateds, gamma=0.99, lambda_=1.0,
                 c_bar=1.0, bootstrap_value=None, truncateds=None, next_values=None, out=None,
                 stream=None):
    N, T, (r, v, q, lr, d) = _prep(rewards, [(values, "values"), (q_values, "q_values"),
                                             (log_rhos, "log_rhos"),
                                             (terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, q, lr, d, tr, nv, b, o, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_retrace(_ptr(r), _ptr(v), _ptr(q), _ptr(lr), _ptr(d), _ptr(tr), _ptr(nv),
                             _ptr(b), _ptr(o), N, T, gamma, lambda_, c_bar, _ptr(ws), wsb,
                             _stream(stream)), "rlcs_retrace")
    return _finish(o, rewards)


def rlcs_eligibility_traces(x, dones, gamma=0.99, lambda_=0.95, out=None, stream=None):
    N, T, (xx, d) = _prep(x, [(dones, "dones")], rewards_name="x")
    o = torch.empty_like(xx) if out is None else _out(out, "out", xx)
    _devices(xx, d, o, stream=stream)
    ws, wsb = workspace_for(N, T, xx.device, stream)
    _check(_lib.rlcs_eligibility_traces(_ptr(xx), _ptr(d), _ptr(o), N, T, gamma, lambda_,
                                        _ptr(ws), wsb, _stream(stream)),
           "rlcs_eligibility_traces")
    return _finish(o, x)


def rlcs_episodic_prefix_sum(x, dones, out=None, stream=None):
    xx = _rows(x, "x", dtype=torch.int32)
    N, T = xx.shape
    d = _rows(dones, "dones")
    if d.shape != (N, T):
        raise ValueError("dones must have shape (%d, %d)" % (N, T))
    o = torch.empty_like(xx) if out is None else _out(out, "out", xx)
    _devices(xx, d, o, stream=stream)
    ws, wsb = workspace_for(N, T, xx.device, stream)
    _check(_lib.rlcs_episodic_prefix_sum(_ptr(xx), _ptr(d), _ptr(o), N, T, _ptr(ws), wsb,
                                         _stream(stream)), "rlcs_episodic_prefix_sum")
    return _finish(o, x)


def rlcs_gae_and_returns(rewards, values, terminateds, gamma=0.99, lambda_=0.95,
                         bootstrap_value=None, truncateds=None, next_values=None, out=None,
                         out_returns=None, stream=None):
    """Returns (advantages, returns) from one pass over the inputs."""
    N, T, (r, v, d) = _prep(rewards, [(values, "values"), (terminateds, "terminateds")])
    tr, nv = _opt(truncateds, "truncateds", N, T), _opt(next_values, "next_values", N, T)
    b = _boot(bootstrap_value, N)
    adv = torch.empty_like(r) if out is None else _out(out, "out", r)
    ret = torch.empty_like(r) if out_returns is None else _out(out_returns, "out_returns", r)
    _devices(r, v, d, tr, nv, b, adv, ret, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_gae_and_returns(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                                     _ptr(adv), _ptr(ret), N, T, gamma, lambda_, _ptr(ws), wsb,
                                     _stream(stream)), "rlcs_gae_and_returns")
    return _finish(adv, rewards), _finish(ret, rewards)


def rlcs_affine_scan(a, b, reset=None, x_init=None, reverse=False, out=None, stream=None):
    """x_t = a_t*x_{t-1} + b_t (reverse: x_t = a_t*x_{t+1} + b_t) per row."""
    N, T, (aa, bb) = _prep(a, [(b, "b")], rewards_name="a")
    rr = _opt(reset, "reset", N, T)
    x0 = None
    if x_init is not None:
        x0 = x_init.reshape(-1)
        if not x0.is_cuda or x0.dtype != torch.float32 or x0.numel() != N:
            raise ValueError("x_init must be a float32 CUDA tensor of %d values" % N)
        x0 = x0.contiguous()
    o = torch.empty_like(aa) if out is None else _out(out, "out", aa)
    _devices(aa, bb, rr, x0, o, stream=stream)
    ws, wsb = workspace_for(N, T, aa.device, stream)
    _check(_lib.rlcs_affine_scan(_ptr(aa), _ptr(bb), _ptr(rr), _ptr(x0), _ptr(o), N, T,
                                 1 if reverse else 0, _ptr(ws), wsb, _stream(stream)),
           "rlcs_affine_scan")
    return _finish(o, a)


def rlcs_gae_compact(rewards, values, terminateds, gamma=0.99, lambda_=0.95,
                     bootstrap_value=None, truncateds=None, next_values=None, out=None,
                     stream=None):
    """GAE from compact inputs: rewards, values, next_values as bf16 bit patterns
    (torch.int16/uint16 or torch.bfloat16 tensors), masks as uint8 (or bool).
    Returns float32 advantages."""
    def bits16(t, name):
        if t is None:
            return None
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        if t.dtype not in (torch.int16, torch.uint16):
            raise TypeError("%s must hold bf16 bit patterns (bfloat16, int16 or uint16)" % name)
        return _rows(t, name, dtype=t.dtype)

    def mask8(t, name):
        if t is None:
            return None
        if t.dtype == torch.bool:
            t = t.view(torch.uint8)
        return _rows(t, name, dtype=torch.uint8)

    r, v = bits16(rewards, "rewards"), bits16(values, "values")
    d = mask8(terminateds, "terminateds")
    N, T = r.shape
    for x, name in ((v, "values"), (d, "terminateds")):
        if x.shape != (N, T):
            raise ValueError("%s must have shape (%d, %d)" % (name, N, T))
    tr, nv = mask8(truncateds, "truncateds"), bits16(next_values, "next_values")
    b = _boot(bootstrap_value, N)
    o = (torch.empty((N, T), dtype=torch.float32, device=r.device) if out is None
         else _out(out, "out", r, dtype=torch.float32))
    _devices(r, v, d, tr, nv, b, o, stream=stream)
    ws, wsb = workspace_for(N, T, r.device, stream)
    _check(_lib.rlcs_gae_compact(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b), _ptr(o),
                                 N, T, gamma, lambda_, _ptr(ws), wsb, _stream(stream)),
           "rlcs_gae_compact")
    return o.reshape(rewards.shape)


def rlcs_diag_stream_copy(inputs, out, empty=False, stream=None):
    """Diagnostic: the warp-row launch shape moving the same bytes as an
    estimator without the scan (sum of the inputs into `out`)."""
    if not isinstance(out, torch.Tensor) or out.dim() != 2 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, T] tensor")
    out = _rows(out, "out")  # device and dtype; already contiguous, so not copied
    N, T = out.shape
    ins = []
    for i, t in enumerate(inputs):
        x = _rows(t, "inputs[%d]" % i)
        if x.shape != (N, T):
            raise ValueError("inputs[%d] must have shape (%d, %d)" % (i, N, T))
        ins.append(x)
    _devices(out, *ins, stream=stream)
    ptrs = (ctypes.c_void_p * len(ins))(*[t.data_ptr() for t in ins])
    _check(_lib.rlcs_diag_stream_copy(ctypes.cast(ptrs, ctypes.c_void_p), len(ins), _ptr(out),
                                      N, T, 1 if empty else 0, _stream(stream)),
           "rlcs_diag_stream_copy")


# ---------------------------------------------------------------------------
# Time-major [T, N] variants: same arguments as above with every per-step
# tensor shaped [T, N]; bootstrap_value / x_init stay [N].
# ---------------------------------------------------------------------------
def _tm_ws(N, T, device, stream):
    return workspace_for(N, T, device, stream, need=_lib.rlcs_workspace_bytes_tm(N, T))


def _tm(*tensors, names, dtypes=None):
    T, N = tensors[0].shape
    out = []
    for i, (t, name) in enumerate(zip(tensors, names)):
        if t is None:
            out.append(None)
            continue
        dt = dtypes[i] if dtypes else torch.float32
        x = _rows(t, name, dtype=dt)
        if x.shape != (T, N):
            raise ValueError("%s must have shape (T=%d, N=%d)" % (name, T, N))
        out.append(x)
    return T, N, out


def rlcs_gae_tm(rewards, values, terminateds, gamma=0.99, lambda_=0.95, bootstrap_value=None,
                truncateds=None, next_values=None, out=None, stream=None):
    T, N, (r, v, d, tr, nv) = _tm(rewards, values, terminateds, truncateds, next_values,
                                  names=("rewards", "values", "terminateds", "truncateds",
                                         "next_values"))
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, d, tr, nv, b, o, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_gae_tm(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b), _ptr(o), N, T,
                            gamma, lambda_, _ptr(ws), wsb, _stream(stream)), "rlcs_gae_tm")
    return o


def rlcs_lambda_returns_tm(rewards, values, terminateds, gamma=0.99, lambda_=0.95,
                           bootstrap_value=None, truncateds=None, next_values=None, out=None,
                           stream=None):
    T, N, (r, v, d, tr, nv) = _tm(rewards, values, terminateds, truncateds, next_values,
                                  names=("rewards", "values", "terminateds", "truncateds",
                                         "next_values"))
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, d, tr, nv, b, o, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_lambda_returns_tm(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                                       _ptr(o), N, T, gamma, lambda_, _ptr(ws), wsb,
                                       _stream(stream)),
           "rlcs_lambda_returns_tm")
    return o


def rlcs_discounted_returns_tm(rewards, terminateds, gamma=0.99, bootstrap_value=None,
                               truncateds=None, next_values=None, out=None, stream=None):
    T, N, (r, d, tr, nv) = _tm(rewards, terminateds, truncateds, next_values,
                               names=("rewards", "terminateds", "truncateds", "next_values"))
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, d, tr, nv, b, o, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_discounted_returns_tm(_ptr(r), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b), _ptr(o),
                                           N, T, gamma, _ptr(ws), wsb, _stream(stream)),
           "rlcs_discounted_returns_tm")
    return o


def rlcs_vtrace_tm(rewards, values, log_rhos, terminateds, gamma=0.99, lambda_=1.0, rho_bar=1.0,
                   c_bar=1.0, bootstrap_value=None, truncateds=None, next_values=None,
                   with_pg=True, out=None, out_pg=None, stream=None):
    T, N, (r, v, lr, d, tr, nv) = _tm(rewards, values, log_rhos, terminateds, truncateds,
                                      next_values,
                                      names=("rewards", "values", "log_rhos", "terminateds",
                                             "truncateds", "next_values"))
    b = _boot(bootstrap_value, N)
    vs = torch.empty_like(r) if out is None else _out(out, "out", r)
    pg = (torch.empty_like(r) if out_pg is None else _out(out_pg, "out_pg", r)) if with_pg else None
    _devices(r, v, lr, d, tr, nv, b, vs, pg, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_vtrace_tm(_ptr(r), _ptr(v), _ptr(lr), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                               _ptr(vs), _ptr(pg), N, T, gamma, lambda_, rho_bar, c_bar,
                               _ptr(ws), wsb, _stream(stream)), "rlcs_vtrace_tm")
    return vs, pg


def rlcs_retrace_tm(rewards, values, q_values, log_rhos, terminateds, gamma=0.99, lambda_=1.0,
                    c_bar=1.0, bootstrap_value=None, truncateds=None, next_values=None, out=None,
                    stream=None):
    T, N, (r, v, q, lr, d, tr, nv) = _tm(rewards, values, q_values, log_rhos, terminateds,
                                         truncateds, next_values,
                                         names=("rewards", "values", "q_values", "log_rhos",
                                                "terminateds", "truncateds", "next_values"))
    b = _boot(bootstrap_value, N)
    o = torch.empty_like(r) if out is None else _out(out, "out", r)
    _devices(r, v, q, lr, d, tr, nv, b, o, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_retrace_tm(_ptr(r), _ptr(v), _ptr(q), _ptr(lr), _ptr(d), _ptr(tr), _ptr(nv),
                                _ptr(b), _ptr(o), N, T, gamma, lambda_, c_bar, _ptr(ws), wsb,
                                _stream(stream)),
           "rlcs_retrace_tm")
    return o


def rlcs_eligibility_traces_tm(x, dones, gamma=0.99, lambda_=0.95, out=None, stream=None):
    T, N, (xx, d) = _tm(x, dones, names=("x", "dones"))
    o = torch.empty_like(xx) if out is None else _out(out, "out", xx)
    _devices(xx, d, o, stream=stream)
    ws, wsb = _tm_ws(N, T, xx.device, stream)
    _check(_lib.rlcs_eligibility_traces_tm(_ptr(xx), _ptr(d), _ptr(o), N, T, gamma, lambda_,
                                           _ptr(ws), wsb, _stream(stream)),
           "rlcs_eligibility_traces_tm")
    return o


def rlcs_episodic_prefix_sum_tm(x, dones, out=None, stream=None):
    T, N, (xx, d) = _tm(x, dones, names=("x", "dones"), dtypes=(torch.int32, torch.float32))
    o = torch.empty_like(xx) if out is None else _out(out, "out", xx)
    _devices(xx, d, o, stream=stream)
    ws, wsb = _tm_ws(N, T, xx.device, stream)
    _check(_lib.rlcs_episodic_prefix_sum_tm(_ptr(xx), _ptr(d), _ptr(o), N, T, _ptr(ws), wsb,
                                            _stream(stream)),
           "rlcs_episodic_prefix_sum_tm")
    return o


def rlcs_gae_and_returns_tm(rewards, values, terminateds, gamma=0.99, lambda_=0.95,
                            bootstrap_value=None, truncateds=None, next_values=None, out=None,
                            out_returns=None, stream=None):
    T, N, (r, v, d, tr, nv) = _tm(rewards, values, terminateds, truncateds, next_values,
                                  names=("rewards", "values", "terminateds", "truncateds",
                                         "next_values"))
    b = _boot(bootstrap_value, N)
    adv = torch.empty_like(r) if out is None else _out(out, "out", r)
    ret = torch.empty_like(r) if out_returns is None else _out(out_returns, "out_returns", r)
    _devices(r, v, d, tr, nv, b, adv, ret, stream=stream)
    ws, wsb = _tm_ws(N, T, r.device, stream)
    _check(_lib.rlcs_gae_and_returns_tm(_ptr(r), _ptr(v), _ptr(d), _ptr(tr), _ptr(nv), _ptr(b),
                                        _ptr(adv), _ptr(ret), N, T, gamma, lambda_,
                                        _ptr(ws), wsb, _stream(stream)), "rlcs_gae_and_returns_tm")
    return adv, ret


def rlcs_affine_scan_tm(a, b, reset=None, x_init=None, reverse=False, out=None, stream=None):
    T, N, (aa, bb, rr) = _tm(a, b, reset, names=("a", "b", "reset"))
    x0 = None if x_init is None else _boot(x_init, N)
    o = torch.empty_like(aa) if out is None else _out(out, "out", aa)
    _devices(aa, bb, rr, x0, o, stream=stream)
    ws, wsb = _tm_ws(N, T, aa.device, stream)
    _check(_lib.rlcs_affine_scan_tm(_ptr(aa), _ptr(bb), _ptr(rr), _ptr(x0), _ptr(o), N, T,
                                    1 if reverse else 0, _ptr(ws), wsb, _stream(stream)),
           "rlcs_affine_scan_tm")
    return o


# ---------------------------------------------------------------------------
# Grouped calls on short rows (T <= 512): one launch per class of calls.
# ---------------------------------------------------------------------------
class RlcsCall(ctypes.Structure):
    """Mirror of rlcs_call in include/rlcs.h."""
    _fields_ = [("estimator", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rewards", ctypes.c_void_p), ("values", ctypes.c_void_p),
                ("q_values", ctypes.c_void_p), ("log_rhos", ctypes.c_void_p),
                ("terminateds", ctypes.c_void_p), ("truncateds", ctypes.c_void_p),
                ("next_values", ctypes.c_void_p), ("bootstrap_value", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("out2", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("T", ctypes.c_int64),
                ("gamma", ctypes.c_double), ("lambda_", ctypes.c_double),
                ("rho_bar", ctypes.c_double), ("c_bar", ctypes.c_double)]


GROUP_ESTIMATORS = {"gae": 0, "lambda_returns": 1, "discounted_returns": 2, "vtrace": 3,
                    "retrace": 4, "eligibility_traces": 5, "episodic_prefix_sum": 6,
                    "gae_and_returns": 7}
MAX_GROUP = 16


def _group_call(est, kw):
    """(RlcsCall, result, tensors to keep alive) for one grouped call; the
    keywords and defaults are those of the namesake wrapper."""
    kw = dict(kw)
    c = RlcsCall()
    c.estimator = GROUP_ESTIMATORS[est]
    keep = []

    def take(name, dtype=torch.float32, required=True):
        t = kw.pop(name, None)
        if t is None:
            if required:
                raise ValueError("%s: %s is required" % (est, name))
            return None
        x = _rows(t, name, dtype)
        keep.append(x)
        return x

    if est in ("eligibility_traces", "episodic_prefix_sum"):
        x = take("x", torch.int32 if est == "episodic_prefix_sum" else torch.float32)
        d = take("dones")
        N, T = x.shape
        if d.shape != (N, T):
            raise ValueError("dones must have shape (%d, %d)" % (N, T))
        c.rewards, c.terminateds = x.data_ptr(), d.data_ptr()
        lead = x
    else:
        r = take("rewards")
        N, T = r.shape
        named = {"values": est != "discounted_returns",
                 "q_values": est == "retrace",
                 "log_rhos": est in ("vtrace", "retrace"),
                 "terminateds": True}
        for name, used in named.items():
            if used:
                t = take(name)
                if t.shape != (N, T):
                    raise ValueError("%s must have shape (%d, %d)" % (name, N, T))
                setattr(c, name, t.data_ptr())
        for name in ("truncateds", "next_values"):
            t = _opt(kw.pop(name, None), name, N, T)
            if t is not None:
                keep.append(t)
                setattr(c, name, t.data_ptr())
        b = _boot(kw.pop("bootstrap_value", None), N)
        if b is not None:
            keep.append(b)
            c.bootstrap_value = b.data_ptr()
        c.rewards = r.data_ptr()
        lead = r
    lam_default = 1.0 if est in ("vtrace", "retrace") else 0.95
    c.gamma = kw.pop("gamma", 0.99)
    c.lambda_ = kw.pop("lambda_", lam_default)
    c.rho_bar = kw.pop("rho_bar", 1.0)
    c.c_bar = kw.pop("c_bar", 1.0)
    c.N, c.T = N, T
    out = kw.pop("out", None)
    out = torch.empty_like(lead) if out is None else _out(out, "out", lead)
    keep.append(out)
    c.out = out.data_ptr()
    result = out
    if est == "vtrace":
        pg = kw.pop("out_pg", None)
        if kw.pop("with_pg", True):
            pg = torch.empty_like(lead) if pg is None else _out(pg, "out_pg", lead)
            keep.append(pg)
            c.out2 = pg.data_ptr()
        else:
            pg = None
        result = (out, pg)
    elif est == "gae_and_returns":
        ret = kw.pop("out_returns", None)
        ret = torch.empty_like(lead) if ret is None else _out(ret, "out_returns", lead)
        keep.append(ret)
        c.out2 = ret.data_ptr()
        result = (out, ret)
    if kw:
        raise TypeError("%s: unexpected arguments %s" % (est, sorted(kw)))
    return c, result, keep


def rlcs_run_group(calls, stream=None):
    """Run estimator calls in one launch per class (short rows by 128 / 256
    / 512 steps, long rows by tile length; truncation inputs present or not).
    `calls` is a list of (estimator, kwargs) pairs: the estimator is a key of
    GROUP_ESTIMATORS and kwargs are what its namesake wrapper takes (x and
    dones for the two forward estimators). Returns the namesakes' results, in
    order. A list longer than MAX_GROUP runs as consecutive groups of
    MAX_GROUP on the same stream. Within a group no output may overlap
    another call's arrays: the calls run concurrently."""
    if len(calls) > MAX_GROUP:
        out = []
        for i in range(0, len(calls), MAX_GROUP):
            out += rlcs_run_group(calls[i:i + MAX_GROUP], stream)
        return out
    arr = (RlcsCall * max(1, len(calls)))()
    keep, results = [], []
    for i, (est, kw) in enumerate(calls):
        c, res, k = _group_call(est, kw)
        arr[i] = c
        keep += k
        results.append(res)
    if keep:
        _devices(keep[0], *keep[1:], stream=stream)
    ptr = ctypes.cast(arr, ctypes.c_void_p)
    need = _lib.rlcs_group_workspace_bytes(ptr, len(calls)) if calls else 0
    ws, wsb = None, 0
    if need:
        ws, wsb = workspace_for(0, 0, keep[0].device, stream, need=need)
    _check(_lib.rlcs_run_group(ptr, len(calls), _ptr(ws), wsb, _stream(stream)),
           "rlcs_run_group")
    return results


def rlcs_check_status(workspace=None, stream=None):
    _check(_lib.rlcs_check_status(_ptr(workspace), _stream(stream)), "rlcs_check_status")


def rlcs_set_shape_override(shape=RLCS_SHAPE_AUTO, chunk=0):
    _check(_lib.rlcs_set_shape_override(shape, chunk), "rlcs_set_shape_override")


def rlcs_workspace_bytes(N, T):
    return _lib.rlcs_workspace_bytes(N, T)


def check_all_workspaces():
    """Synchronise and check the status word of every cached workspace."""
    with _ws_lock:
        items = list(_ws_cache.values())
    for ws in items:
        _check(_lib.rlcs_check_status(_ptr(ws), None), "rlcs_check_status")
