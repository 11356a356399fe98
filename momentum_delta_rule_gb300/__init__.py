"""Momentum DeltaNet (MDN) memory update on GB300 — Python binding.

A thin ctypes layer over the C ABI in ``include/mdn.h`` (``libmdn.so``, built
in-tree by ``momentum_delta_rule_gb300.build``).  It only marshals arguments:
checks dtypes, devices and contiguity, allocates outputs and the workspace
with PyTorch, passes raw device pointers and the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no
other code path.  If the library is missing, every call raises.

Entry points (same names as the C ABI):
  chunk_fwd(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
            cu_seqlens=None, ...)               -> (o, S_T, M_T)
            (return_vres=True: (o, S_T, M_T, vres) via mdn_chunk_fwd_vres;
             return_chunk_states=True: (o, S_T, M_T, S_chunks, M_chunks)
             via mdn_chunk_fwd_states)
  chunk_state_slots(n_seq, B, T, packed)
  decode_step(q, k, v, alpha, mu, eta, S, M, beta=None, o=None) -> o
  prepare_inputs(q, k, z_alpha, z_beta, z_mu, z_eta, a, b, s, tau,
                 log_mu_min=-2.0, comba_d=0.0) -> (q_hat, k_hat, alpha, beta, mu, eta)
  workspace_size(n_seq, T_total, H, D, dtype)
  device_status(stream=None), wait_selftest(limit_us), abi_version(),
  status_string(code)
"""
import ctypes
import os

import torch

__all__ = ["chunk_fwd", "chunk_fwd_kernel_count", "chunk_bwd", "block_fwd", "chunk_bwd_workspace_size", "chunk_state_slots", "decode_step", "prepare_inputs", "workspace_size",
           "device_status", "wait_selftest",
           "abi_version", "status_string", "MdnError", "lib", "LIB_PATH",
           "EXPORTED_SYMBOLS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmdn.so")

MDN_OK = 0
MDN_ERR_INVALID_ARG = 1
MDN_ERR_UNSUPPORTED = 2
MDN_ERR_CUDA = 3
MDN_ERR_DEVICE_TIMEOUT = 4
MDN_F32 = 0
MDN_BF16 = 1
CHUNK = 64

EXPORTED_SYMBOLS = ["mdn_abi_version", "mdn_status_string",
                    "mdn_chunk_fwd_workspace_size", "mdn_chunk_fwd",
                    "mdn_chunk_fwd_profiled", "mdn_chunk_fwd_static_ws",
                    "mdn_chunk_fwd_vres", "mdn_chunk_state_slots",
                    "mdn_chunk_fwd_states", "mdn_prepare_inputs",
                    "mdn_decode_step", "mdn_get_device_status",
                    "mdn_wait_selftest", "mdn_chunk_bwd_workspace_size",
                    "mdn_chunk_bwd", "mdn_block_fwd_workspace_size", "mdn_block_fwd",
                    "mdn_chunk_fwd_kernel_count"]
MDN_PATH_CUDA_CORE = 0
MDN_PATH_TENSOR_CORE = 1

_LIB = None


class MdnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def lib():
    """Load ``libmdn.so`` once; raise if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libmdn.so not found at %s; build it with "
            "`python -m momentum_delta_rule_gb300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    c_int, c_size = ctypes.c_int, ctypes.c_size_t
    L.mdn_abi_version.restype = c_int
    L.mdn_abi_version.argtypes = []
    L.mdn_status_string.restype = ctypes.c_char_p
    L.mdn_status_string.argtypes = [c_int]
    L.mdn_chunk_fwd_workspace_size.restype = c_size
    L.mdn_chunk_fwd_workspace_size.argtypes = [c_int] * 5 + [c_int]
    L.mdn_chunk_fwd_kernel_count.restype = c_int
    L.mdn_chunk_fwd_kernel_count.argtypes = [c_int] * 9
    L.mdn_chunk_fwd.restype = c_int
    L.mdn_chunk_fwd.argtypes = ([vp] * 3 + [fp] * 6 + [vp, fp, fp, ip]
                                + [c_int] * 8 + [vp, c_size, vp])
    L.mdn_chunk_fwd_profiled.restype = c_int
    L.mdn_chunk_fwd_profiled.argtypes = (L.mdn_chunk_fwd.argtypes
                                         + [ctypes.POINTER(ctypes.c_void_p), c_int,
                                            ctypes.POINTER(ctypes.c_int)])
    L.mdn_chunk_fwd_vres.restype = c_int
    L.mdn_chunk_fwd_vres.argtypes = ([vp] * 3 + [fp] * 6 + [vp, fp, fp, vp, ip]
                                     + [c_int] * 8 + [vp, c_size, vp])
    L.mdn_chunk_state_slots.restype = c_size
    L.mdn_chunk_state_slots.argtypes = [c_int] * 4
    L.mdn_chunk_fwd_states.restype = c_int
    L.mdn_chunk_fwd_states.argtypes = ([vp] * 3 + [fp] * 6 + [vp, fp, fp, fp, fp, ip]
                                       + [c_int] * 8 + [vp, c_size, vp])
    L.mdn_chunk_fwd_static_ws.restype = c_int
    L.mdn_chunk_fwd_static_ws.argtypes = ([vp] * 3 + [fp] * 6 + [vp, fp, fp, ip]
                                          + [c_int] * 8 + [vp])
    L.mdn_decode_step.restype = c_int
    L.mdn_decode_step.argtypes = [vp] * 3 + [fp] * 6 + [vp] + [c_int] * 5 + [vp]
    L.mdn_prepare_inputs.restype = c_int
    c_float = ctypes.c_float
    L.mdn_prepare_inputs.argtypes = ([vp] * 2 + [fp] * 4 + [vp] * 2 + [fp] * 4
                                     + [c_int] * 4 + [c_float] * 6 + [vp])
    L.mdn_get_device_status.restype = c_int
    L.mdn_get_device_status.argtypes = [vp]
    L.mdn_wait_selftest.restype = c_int
    L.mdn_wait_selftest.argtypes = [c_int, vp]
    L.mdn_block_fwd_workspace_size.restype = c_size
    L.mdn_block_fwd_workspace_size.argtypes = [c_int] * 6
    c_float = ctypes.c_float
    L.mdn_block_fwd.restype = c_int
    L.mdn_block_fwd.argtypes = ([vp] * 5 + [c_float] * 7 + [vp] * 6 + [c_int] * 7
                                + [vp, c_size, vp])
    L.mdn_chunk_bwd_workspace_size.restype = c_size
    L.mdn_chunk_bwd_workspace_size.argtypes = [c_int] * 6
    L.mdn_chunk_bwd.restype = c_int
    L.mdn_chunk_bwd.argtypes = [vp] * 23 + [c_int] * 8 + [vp, c_size, vp]
    _LIB = L
    return L


def abi_version():
    return lib().mdn_abi_version()


def status_string(code):
    try:
        return lib().mdn_status_string(int(code)).decode()
    except RuntimeError:
        return "status %d" % code


def _dtype_code(t):
    if t == torch.bfloat16:
        return MDN_BF16
    if t == torch.float32:
        return MDN_F32
    raise TypeError("q/k/v must be float32 or bfloat16, got %s" % t)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(name, t, dtype=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def workspace_size(n_seq, T_total, H, D, dtype):
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().mdn_chunk_fwd_workspace_size(n_seq, T_total, H, D, D, code))


def chunk_fwd_kernel_count(n_seq, B, T, H, D, dtype, packed, final_states=True):
    """Kernels one ``chunk_fwd`` call with these sizes enqueues on the current
    device (``mdn_chunk_fwd_kernel_count``); 0 for rejected sizes."""
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().mdn_chunk_fwd_kernel_count(int(n_seq), int(B), int(T), int(H), int(D),
                                                int(D), code, 1 if packed else 0,
                                                1 if final_states else 0))


def chunk_fwd(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
              cu_seqlens=None, o=None, S_T=None, M_T=None,
              output_final_state=True, workspace=None, stream=None,
              stage_events=None, info=None, return_vres=False, vres=None,
              return_chunk_states=False, S_chunks=None, M_chunks=None):
    """Prefill over whole sequences (``mdn_chunk_fwd``).

    q, k ``[B, T, H, D]`` and v ``[B, T, H, D]`` (fp32 or bf16, same dtype);
    gates ``[B, T, H]`` fp32; S0/M0 ``[n_seq, H, D, D]`` fp32 or None;
    ``cu_seqlens`` int32 CUDA tensor ``[n_seq + 1]`` for packed sequences
    (then B == 1).  Returns ``(o, S_T, M_T)``; the states are None when
    ``output_final_state`` is False.  With ``return_vres`` (or a ``vres``
    buffer shaped like v) the per-token residuals come fourth.  With
    ``return_chunk_states`` (or ``S_chunks``/``M_chunks`` buffers of
    ``[chunk_state_slots(...), H, D, D]`` in the dtype of q) the entry
    states of every chunk come fourth and fifth (``mdn_chunk_fwd_states``;
    bf16 for bf16 inputs, as the gradient pass reads them).
    """
    L = lib()
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, D]")
    B, T, H, D = q.shape
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype, dev)
        if tuple(t.shape) != (B, T, H, D):
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), (B, T, H, D)))
    for name, t in (("alpha", alpha), ("mu", mu), ("eta", eta), ("beta", beta)):
        if name != "beta" and t is None:
            raise ValueError("%s is required" % name)
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (B, T, H):
            raise ValueError("%s must be [B, T, H]" % name)
    if cu_seqlens is not None:
        _check_cuda("cu_seqlens", cu_seqlens, torch.int32, dev)
        n_seq = cu_seqlens.numel() - 1
    else:
        n_seq = B
    for name, t in (("S0", S0), ("M0", M0)):
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (n_seq, H, D, D):
            raise ValueError("%s must be [n_seq, H, D, D]" % name)
    if o is None:
        o = torch.empty_like(v)
    _check_cuda("o", o, q.dtype, dev)
    if output_final_state:
        if S_T is None:
            S_T = torch.empty((n_seq, H, D, D), dtype=torch.float32, device=dev)
        if M_T is None:
            M_T = torch.empty((n_seq, H, D, D), dtype=torch.float32, device=dev)
    _check_cuda("S_T", S_T, torch.float32, dev)
    _check_cuda("M_T", M_T, torch.float32, dev)
    want_vres = return_vres or vres is not None
    if want_vres:
        if stage_events is not None or info is not None:
            raise ValueError("stage_events/info are not available with the residual output")
        if vres is None:
            vres = torch.empty_like(v)
        _check_cuda("vres", vres, q.dtype, dev)
        if tuple(vres.shape) != (B, T, H, D):
            raise ValueError("vres must have the shape of v")
    want_states = return_chunk_states or S_chunks is not None or M_chunks is not None
    if want_states:
        if want_vres or stage_events is not None or info is not None:
            raise ValueError("the chunk states come alone, without residuals or stage events")
        slots = chunk_state_slots(n_seq, B, T, cu_seqlens is not None)
        for name in ("S_chunks", "M_chunks"):
            t = S_chunks if name == "S_chunks" else M_chunks
            if t is None:
                t = torch.empty((max(slots, 1), H, D, D), dtype=q.dtype, device=dev)
            _check_cuda(name, t, q.dtype, dev)
            if t.dim() != 4 or t.shape[0] < slots or tuple(t.shape[1:]) != (H, D, D):
                raise ValueError("%s must be [>= %d, H, D, D]" % (name, slots))
            if name == "S_chunks":
                S_chunks = t
            else:
                M_chunks = t
    need = int(L.mdn_chunk_fwd_workspace_size(n_seq, B * T, H, D, D, code))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, torch.uint8, dev)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(mu), _ptr(eta),
            _ptr(beta), _ptr(S0), _ptr(M0), _ptr(o), _ptr(S_T), _ptr(M_T),
            _ptr(cu_seqlens), n_seq, B, T, H, D, D, code, CHUNK,
            _ptr(workspace), workspace.numel(), _stream_handle(dev, stream))
    with torch.cuda.device(dev):
        if want_states:
            st = L.mdn_chunk_fwd_states(*(args[:12] + (_ptr(S_chunks), _ptr(M_chunks)) + args[12:]))
            if st != MDN_OK:
                raise MdnError(st, "mdn_chunk_fwd_states")
            return o, S_T, M_T, S_chunks, M_chunks
        if want_vres:
            st = L.mdn_chunk_fwd_vres(*(args[:12] + (_ptr(vres),) + args[12:]))
            if st != MDN_OK:
                raise MdnError(st, "mdn_chunk_fwd_vres")
            return o, S_T, M_T, vres
        if stage_events is None and info is None:
            st = L.mdn_chunk_fwd(*args)
        else:
            n_ev = 0 if stage_events is None else len(stage_events)
            for e in (stage_events or []):
                if e.cuda_event == 0:       # torch creates events lazily
                    e.record(torch.cuda.current_stream(dev) if stream is None else stream)
            arr = (ctypes.c_void_p * max(n_ev, 1))(
                *[ctypes.c_void_p(e.cuda_event) for e in (stage_events or [])])
            path = ctypes.c_int(-1)
            st = L.mdn_chunk_fwd_profiled(*args, arr if n_ev else None, n_ev,
                                          ctypes.byref(path))
            if info is not None:
                info["path"] = path.value
    if st != MDN_OK:
        raise MdnError(st, "mdn_chunk_fwd")
    return o, S_T, M_T


def chunk_state_slots(n_seq, B, T, packed):
    """Chunk slots the entry-state outputs need (``mdn_chunk_state_slots``):
    chunk c of sequence s at slot s * ceil(T / 64) + c, or, packed, at
    sum_{s' < s} ceil(L_s' / 64) + c."""
    return int(lib().mdn_chunk_state_slots(int(n_seq), int(B), int(T), 1 if packed else 0))


def decode_step(q, k, v, alpha, mu, eta, S, M, beta=None, o=None, stream=None):
    """One recurrent step per sequence (``mdn_decode_step``), S and M in place.

    q, k, v ``[N, H, D]``; gates ``[N, H]`` fp32; S, M ``[N, H, D, D]`` fp32.
    Returns o ``[N, H, D]`` in the dtype of q.
    """
    L = lib()
    if q.dim() != 3:
        raise ValueError("q must be [N, H, D]")
    N, H, D = q.shape
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype, dev)
        if tuple(t.shape) != (N, H, D):
            raise ValueError("%s must be [N, H, D]" % name)
    for name, t in (("alpha", alpha), ("mu", mu), ("eta", eta), ("beta", beta)):
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (N, H):
            raise ValueError("%s must be [N, H]" % name)
    for name, t in (("S", S), ("M", M)):
        _check_cuda(name, t, torch.float32, dev)
        if tuple(t.shape) != (N, H, D, D):
            raise ValueError("%s must be [N, H, D, D]" % name)
    if o is None:
        o = torch.empty_like(v)
    _check_cuda("o", o, q.dtype, dev)
    with torch.cuda.device(dev):
        st = L.mdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(mu),
                               _ptr(eta), _ptr(beta), _ptr(S), _ptr(M), _ptr(o),
                               N, H, D, D, code, _stream_handle(dev, stream))
    if st != MDN_OK:
        raise MdnError(st, "mdn_decode_step")
    return o


def prepare_inputs(q, k, z_alpha, z_beta, z_mu, z_eta, a, b, s, tau,
                   log_mu_min=-2.0, comba_d=0.0, q_out=None, k_out=None, stream=None):
    """Gates from their projections and normalised q, k (``mdn_prepare_inputs``).

    q, k ``[..., H, d]`` (fp32 or bf16, same dtype; the leading dims are the
    tokens); z_* ``[..., H]`` fp32.  Returns ``(q_hat, k_hat, alpha, beta, mu,
    eta)``; q_out / k_out may be q / k for in-place normalisation.
    """
    L = lib()
    if q.dim() < 2:
        raise ValueError("q must be [..., H, d]")
    H, D = q.shape[-2], q.shape[-1]
    dev = q.device
    code = _dtype_code(q.dtype)
    _check_cuda("q", q, q.dtype, dev)
    _check_cuda("k", k, q.dtype, dev)
    if k.shape != q.shape:
        raise ValueError("k must have the shape of q")
    n_tokens = q.numel() // (H * D)
    for name, t in (("z_alpha", z_alpha), ("z_beta", z_beta), ("z_mu", z_mu), ("z_eta", z_eta)):
        _check_cuda(name, t, torch.float32, dev)
        if tuple(t.shape) != tuple(q.shape[:-1]):
            raise ValueError("%s must be shaped like q without its last dimension" % name)
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    _check_cuda("q_out", q_out, q.dtype, dev)
    _check_cuda("k_out", k_out, q.dtype, dev)
    gates = [torch.empty(q.shape[:-1], dtype=torch.float32, device=dev) for _ in range(4)]
    with torch.cuda.device(dev):
        st = L.mdn_prepare_inputs(_ptr(q), _ptr(k), _ptr(z_alpha), _ptr(z_beta), _ptr(z_mu),
                                  _ptr(z_eta), _ptr(q_out), _ptr(k_out), *[_ptr(g) for g in gates],
                                  n_tokens, H, D, code, float(a), float(b), float(s),
                                  float(tau), float(log_mu_min), float(comba_d),
                                  _stream_handle(dev, stream))
    if st != MDN_OK:
        raise MdnError(st, "mdn_prepare_inputs")
    return (q_out, k_out) + tuple(gates)


def chunk_bwd(q, k, v, alpha, mu, eta, S_chunks, M_chunks, dout, beta=None,
              dS_T=None, dM_T=None, cu_seqlens=None, need_dbeta=True,
              need_dstates=True, workspace=None, stream=None, fwd_workspace=None):
    """Gradients of the chunk forward (``mdn_chunk_bwd``).

    Inputs as ``chunk_fwd`` plus the forward's chunk entry states
    ``S_chunks``, ``M_chunks`` (``chunk_fwd(..., return_chunk_states=True)``),
    the adjoint ``dout`` of o and optionally ``dS_T``, ``dM_T``.
    ``fwd_workspace``: the uint8 workspace the state-saving forward used for
    these inputs, unchanged since (bf16 inputs: its T and A_O T are reused),
    or None.  Returns a dict with dq, dk, dv (dtype of q), dalpha, dmu,
    deta, dbeta (fp32, dbeta None unless ``need_dbeta``), dS0, dM0 (None
    unless ``need_dstates``).
    """
    L = lib()
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, D]")
    B, T, H, D = q.shape
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _check_cuda(name, t, q.dtype, dev)
        if tuple(t.shape) != (B, T, H, D):
            raise ValueError("%s must be [B, T, H, D]" % name)
    for name, t in (("alpha", alpha), ("mu", mu), ("eta", eta), ("beta", beta)):
        if name != "beta" and t is None:
            raise ValueError("%s is required" % name)
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (B, T, H):
            raise ValueError("%s must be [B, T, H]" % name)
    if cu_seqlens is not None:
        _check_cuda("cu_seqlens", cu_seqlens, torch.int32, dev)
        n_seq = cu_seqlens.numel() - 1
    else:
        n_seq = B
    slots = chunk_state_slots(n_seq, B, T, cu_seqlens is not None)
    for name, t in (("S_chunks", S_chunks), ("M_chunks", M_chunks)):
        _check_cuda(name, t, q.dtype, dev)
        if t.dim() != 4 or t.shape[0] < slots or tuple(t.shape[1:]) != (H, D, D):
            raise ValueError("%s must be [>= %d, H, D, D]" % (name, slots))
    if fwd_workspace is not None:
        _check_cuda("fwd_workspace", fwd_workspace, torch.uint8, dev)
        fneed = int(L.mdn_chunk_fwd_workspace_size(n_seq, B * T, H, D, D, code))
        if fwd_workspace.numel() < fneed:
            raise ValueError("fwd_workspace must hold %d bytes" % fneed)
    for name, t in (("dS_T", dS_T), ("dM_T", dM_T)):
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (n_seq, H, D, D):
            raise ValueError("%s must be [n_seq, H, D, D]" % name)
    g = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
         "dalpha": torch.empty_like(alpha), "dmu": torch.empty_like(alpha),
         "deta": torch.empty_like(alpha),
         "dbeta": torch.empty_like(alpha) if need_dbeta else None,
         "dS0": (torch.empty((n_seq, H, D, D), dtype=torch.float32, device=dev)
                 if need_dstates else None)}
    g["dM0"] = torch.empty_like(g["dS0"]) if need_dstates else None
    need = int(L.mdn_chunk_bwd_workspace_size(n_seq, B * T, H, D, D, code))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, torch.uint8, dev)
    with torch.cuda.device(dev):
        st = L.mdn_chunk_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(mu), _ptr(eta), _ptr(beta),
            _ptr(S_chunks), _ptr(M_chunks), _ptr(fwd_workspace), _ptr(dout), _ptr(dS_T), _ptr(dM_T),
            _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dalpha"]), _ptr(g["dmu"]),
            _ptr(g["deta"]), _ptr(g["dbeta"]), _ptr(g["dS0"]), _ptr(g["dM0"]),
            _ptr(cu_seqlens), n_seq, B, T, H, D, D, code, CHUNK, _ptr(workspace),
            workspace.numel(), _stream_handle(dev, stream))
    if st != MDN_OK:
        raise MdnError(st, "mdn_chunk_bwd")
    return g


def block_fwd(x, W_in, conv_w, rms_w, W_o, H, d, a, b, s, tau, log_mu_min=-2.0,
              comba_d=0.0, rms_eps=1e-6, S0=None, M0=None, cu_seqlens=None,
              output_final_state=True, workspace=None, stream=None):
    """The MDN token-mixer block (``mdn_block_fwd``): x ``[B, T, d_model]``
    (or packed ``[1, sum T, d_model]`` with ``cu_seqlens``), weights as the
    header describes.  Returns ``(y, S_T, M_T)``."""
    L = lib()
    if x.dim() != 3:
        raise ValueError("x must be [B, T, d_model]")
    B, T, d_model = x.shape
    dev = x.device
    code = _dtype_code(x.dtype)
    n_cols = 4 * H * d + 4 * H
    for name, t, shape, dt in (("x", x, (B, T, d_model), x.dtype),
                               ("W_in", W_in, (d_model, n_cols), x.dtype),
                               ("conv_w", conv_w, (3 * H * d, 4), torch.float32),
                               ("rms_w", rms_w, (d,), torch.float32),
                               ("W_o", W_o, (H * d, d_model), x.dtype)):
        _check_cuda(name, t, dt, dev)
        if tuple(t.shape) != shape:
            raise ValueError("%s must be %s" % (name, shape))
    if cu_seqlens is not None:
        _check_cuda("cu_seqlens", cu_seqlens, torch.int32, dev)
        n_seq = cu_seqlens.numel() - 1
    else:
        n_seq = B
    for name, t in (("S0", S0), ("M0", M0)):
        _check_cuda(name, t, torch.float32, dev)
        if t is not None and tuple(t.shape) != (n_seq, H, d, d):
            raise ValueError("%s must be [n_seq, H, d, d]" % name)
    y = torch.empty_like(x)
    S_T = M_T = None
    if output_final_state:
        S_T = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
        M_T = torch.empty_like(S_T)
    need = int(L.mdn_block_fwd_workspace_size(n_seq, B * T, H, d, d_model, code))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, torch.uint8, dev)
    with torch.cuda.device(dev):
        st = L.mdn_block_fwd(_ptr(x), _ptr(W_in), _ptr(conv_w), _ptr(rms_w), _ptr(W_o),
                             float(a), float(b), float(s), float(tau), float(log_mu_min),
                             float(comba_d), float(rms_eps), _ptr(S0), _ptr(M0), _ptr(y),
                             _ptr(S_T), _ptr(M_T), _ptr(cu_seqlens), n_seq, B, T, H, d,
                             d_model, code, _ptr(workspace), workspace.numel(),
                             _stream_handle(dev, stream))
    if st != MDN_OK:
        raise MdnError(st, "mdn_block_fwd")
    return y, S_T, M_T


def block_fwd_workspace_size(n_seq, T_total, H, d, d_model, dtype):
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().mdn_block_fwd_workspace_size(n_seq, T_total, H, d, d_model, code))


def chunk_bwd_workspace_size(n_seq, T_total, H, D, dtype):
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().mdn_chunk_bwd_workspace_size(n_seq, T_total, H, D, D, code))


def wait_selftest(limit_us=2000, stream=None, device=None):
    """Enqueue the library's bounded-wait self-test (a kernel waiting on a
    barrier nothing arrives at, for ``limit_us`` microseconds); a later
    ``device_status()`` reports ``MDN_ERR_DEVICE_TIMEOUT``."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = lib().mdn_wait_selftest(int(limit_us), _stream_handle(dev, stream))
    if st != MDN_OK:
        raise MdnError(st, "mdn_wait_selftest")


def device_status(stream=None, device=None):
    """Synchronise and read/clear the device status word (``MDN_OK`` = 0)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return lib().mdn_get_device_status(_stream_handle(dev, stream))
