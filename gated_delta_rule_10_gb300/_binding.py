"""ctypes binding of libgdr.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor devices, dtypes and layouts, allocates outputs with PyTorch and
passes raw pointers plus the current CUDA stream through the C ABI declared in
``include/gdr.h``. There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_F32 = 0
GDR_BF16 = 1
DECAY_CHANNEL = 1
ERASE_CHANNEL = 2
WRITE_CHANNEL = 4
QMIX = 8
BETA_CHANNEL = 16
CHUNK = 64

STATUS = {0: "GDR_OK", 1: "GDR_ERR_INVALID_ARG", 2: "GDR_ERR_UNSUPPORTED", 3: "GDR_ERR_CUDA",
          4: "GDR_ERR_WORKSPACE", 5: "GDR_ERR_TIMEOUT"}


class GdrError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s" % (where, status_string(code)))


class Shape(ctypes.Structure):
    """Mirror of ``gdr_shape``."""
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint), ("scale", ctypes.c_float)]


class OutGate(ctypes.Structure):
    """Mirror of ``gdr_out_gate``."""
    _fields_ = [("z", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("eps", ctypes.c_float)]


_lib = None
_vp = ctypes.c_void_p


def lib():
    """The loaded libgdr.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgdr.so is not built (%s); run __graft_entry__.build() or "
                               "python -m gated_delta_rule_10_gb300.build" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        sp = ctypes.POINTER(Shape)
        L.gdr_chunk_fwd_workspace.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_chunk_fwd_workspace_min.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_chunk_fwd.argtypes = [sp] + [_vp] * 11 + [_vp, ctypes.c_size_t, _vp]
        L.gdr_chunk_fwd_split.argtypes = ([sp, ctypes.c_int] + [_vp] * 11 +
                                          [_vp, ctypes.c_size_t, _vp])
        L.gdr_chunk_fwd_workspace_split.argtypes = [sp, ctypes.c_int,
                                                    ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_chunk_fwd_pipelined.argtypes = ([sp, ctypes.c_int] + [_vp] * 11 +
                                              [_vp, ctypes.c_size_t, _vp, _vp])
        L.gdr_chunk_fwd_workspace_pipelined.argtypes = [sp, ctypes.c_int,
                                                        ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_chunk_fwd_pipeline_segments.argtypes = [sp, ctypes.POINTER(ctypes.c_int)]
        L.gdr_recurrent_step.argtypes = [sp] + [_vp] * 10 + [_vp]
        L.gdr_gate_cumsum.argtypes = [ctypes.c_int] * 4 + [_vp, _vp, _vp]
        L.gdr_chunk_fwd_check.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
        L.gdr_chunk_bwd_check.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
        L.gdr_chunk_bwd_workspace.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_chunk_bwd.argtypes = [sp] + [_vp] * 20 + [_vp, ctypes.c_size_t, _vp]
        L.gdr_token_bwd_workspace.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t)]
        L.gdr_token_bwd.argtypes = [sp] + [_vp] * 20 + [_vp, ctypes.c_size_t, _vp]
        L.gdr_rmsnorm_gate.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                       _vp, ctypes.c_float, _vp, _vp]
        L.gdr_token_fwd.argtypes = [sp] + [_vp] * 11 + [_vp]
        gp = ctypes.POINTER(OutGate)
        L.gdr_chunk_fwd_gated.argtypes = ([sp] + [_vp] * 9 + [gp, _vp, _vp] +
                                          [_vp, ctypes.c_size_t, _vp])
        L.gdr_chunk_fwd_gated_pipelined.argtypes = ([sp, ctypes.c_int] + [_vp] * 9 +
                                                    [gp, _vp, _vp] +
                                                    [_vp, ctypes.c_size_t, _vp, _vp])
        L.gdr_status_string.argtypes = [ctypes.c_int]
        L.gdr_status_string.restype = ctypes.c_char_p
        L.gdr_abi_version.restype = ctypes.c_int
        for name in ("gdr_chunk_fwd_workspace", "gdr_chunk_fwd_workspace_min", "gdr_chunk_fwd",
                     "gdr_chunk_fwd_split", "gdr_chunk_fwd_workspace_split",
                     "gdr_chunk_fwd_pipelined", "gdr_chunk_fwd_workspace_pipelined",
                     "gdr_chunk_fwd_pipeline_segments", "gdr_recurrent_step",
                     "gdr_gate_cumsum", "gdr_chunk_fwd_check", "gdr_chunk_bwd_check", "gdr_rmsnorm_gate",
                     "gdr_chunk_bwd_workspace", "gdr_chunk_bwd", "gdr_token_bwd_workspace", "gdr_token_bwd", "gdr_chunk_fwd_gated",
                     "gdr_chunk_fwd_gated_pipelined", "gdr_token_fwd"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code):
    return lib().gdr_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return _vp(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(t, name, dtype, device, shape=None):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError("%s must be a CUDA tensor on %s" % (name, device))
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def _infer_flags(channel_decay, b, w, lam, channel_beta=False):
    """Variant flags implied by which gates the caller passed."""
    flags = DECAY_CHANNEL if channel_decay else 0
    if channel_beta:
        flags |= BETA_CHANNEL
    if b is not None:
        flags |= ERASE_CHANNEL
    if w is not None:
        flags |= WRITE_CHANNEL
    if lam is not None:
        flags |= QMIX
    return flags


def make_shape(B, T, H, dk, dv, dtype, flags, scale):
    return Shape(B, T, H, dk, dv, GDR_BF16 if dtype == torch.bfloat16 else GDR_F32,
                 flags, float(scale))


def chunk_fwd_workspace_bytes(shape, minimum=False, segments=None):
    """Workspace bytes for a chunk_fwd call on `shape`: the size that selects the
    fastest path, with minimum=True the least the call accepts, or with
    `segments` the size a split into that many runs needs."""
    n = ctypes.c_size_t(0)
    if segments is not None:
        st = lib().gdr_chunk_fwd_workspace_split(ctypes.byref(shape), int(segments), ctypes.byref(n))
        if st:
            raise GdrError(st, "gdr_chunk_fwd_workspace_split")
        return n.value
    name = "gdr_chunk_fwd_workspace_min" if minimum else "gdr_chunk_fwd_workspace"
    st = getattr(lib(), name)(ctypes.byref(shape), ctypes.byref(n))
    if st:
        raise GdrError(st, name)
    return n.value


def pipeline_segments(shape):
    """Time segments ``gdr_chunk_fwd_pipelined`` should use on `shape` (1: none)."""
    n = ctypes.c_int(1)
    st = lib().gdr_chunk_fwd_pipeline_segments(ctypes.byref(shape), ctypes.byref(n))
    if st:
        raise GdrError(st, "gdr_chunk_fwd_pipeline_segments")
    return n.value


def chunk_fwd_pipelined_workspace_bytes(shape, segments):
    n = ctypes.c_size_t(0)
    st = lib().gdr_chunk_fwd_workspace_pipelined(ctypes.byref(shape), int(segments),
                                                 ctypes.byref(n))
    if st:
        raise GdrError(st, "gdr_chunk_fwd_workspace_pipelined")
    return n.value


_aux_streams = {}


def aux_stream(device):
    """The high-priority stream of `device` that pipelined forwards run their
    state passes on (created once per device)."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    if idx not in _aux_streams:
        _aux_streams[idx] = torch.cuda.Stream(device=idx, priority=-1)
    return _aux_streams[idx]


def chunk_fwd(q, k, v, g, beta=None, lam=None, b=None, w=None, h0=None, *, scale=None,
              flags=None, output_final_state=True, o=None, hT=None, workspace=None,
              segments=None, pipeline=None, aux=None, stream=None, out_gate=None):
    """Chunkwise forward (``gdr_chunk_fwd``).

    q, k: [B, T, H, d_k]; v: [B, T, H, d_v] (bf16 or fp32, one dtype);
    g: [B, T, H] or [B, T, H, d_k] fp32 log-decay; beta / lam: [B, T, H] fp32
    (beta [B, T, H, d_v] selects the write strength per value channel);
    b: [B, T, H, d_k]; w: [B, T, H, d_v]; h0: [B, H, d_k, d_v] fp32 or None.
    ``flags`` defaults to what the given gates imply (channel g, b, w, lam);
    ``scale`` to d_k^-1/2. ``workspace`` defaults to the size of the fastest path
    (pass a smaller tensor, even an empty one, to select another path).
    ``segments`` cuts every sequence into that many runs
    (``gdr_chunk_fwd_split``); by default the library decides. ``pipeline``
    runs ``gdr_chunk_fwd_pipelined`` with that many time segments, the state
    passes on ``aux`` (default: this module's high-priority auxiliary stream of
    the device; 1: off); by default (no ``workspace`` or ``segments`` given) the
    library's recommendation is taken. ``out_gate=(z, weight, eps)`` applies the
    output epilogue (``gdr_chunk_fwd_gated``): o then holds y = RMSNorm(o) *
    weight * silu(z) per (token, head) row, z of o's shape and dtype, weight
    [d_v] fp32. Returns (o, hT) with hT None unless requested.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must be bf16 or fp32")
    if flags is None:
        flags = _infer_flags(g.dim() == 4, b, w, lam, beta is not None and beta.dim() == 4)
    if scale is None:
        scale = dk ** -0.5
    _check(q, "q", dt, dev, (B, T, H, dk))
    _check(k, "k", dt, dev, (B, T, H, dk))
    _check(v, "v", dt, dev, (B, T, H, dv))
    _check(g, "g", torch.float32, dev, (B, T, H, dk) if flags & DECAY_CHANNEL else (B, T, H))
    _check(beta, "beta", torch.float32, dev,
           (B, T, H, dv) if flags & BETA_CHANNEL else (B, T, H))
    _check(lam, "lam", torch.float32, dev, (B, T, H))
    _check(b, "b", dt, dev, (B, T, H, dk))
    _check(w, "w", dt, dev, (B, T, H, dv))
    _check(h0, "h0", torch.float32, dev, (B, H, dk, dv))
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=dt, device=dev)
    _check(o, "o", dt, dev, (B, T, H, dv))
    if hT is None and output_final_state:
        hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    _check(hT, "hT", torch.float32, dev, (B, H, dk, dv))
    shape = make_shape(B, T, H, dk, dv, dt, flags, scale)
    if pipeline is None:
        pipeline = (pipeline_segments(shape) if workspace is None and segments is None else 1)
    if pipeline > 1:
        if segments is not None:
            raise ValueError("pipeline and segments select different paths")
        ws_bytes = chunk_fwd_pipelined_workspace_bytes(shape, pipeline)
    else:
        ws_bytes = chunk_fwd_workspace_bytes(shape, segments=segments)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if out_gate is not None:
        z, weight, eps = out_gate
        _check(z, "z", dt, dev, (B, T, H, dv))
        _check(weight, "weight", torch.float32, dev, (dv,))
        if segments is not None and segments != 1:
            raise ValueError("out_gate takes the default or the pipelined path")
        gate = OutGate(_ptr(z), _ptr(weight), float(eps))
        ins = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam), _ptr(b), _ptr(w),
               _ptr(h0))
        tail = (_ptr(o), _ptr(hT), _ptr(workspace),
                ctypes.c_size_t(0 if workspace is None else workspace.numel()),
                _stream(stream, dev))
        with torch.cuda.device(dev):
            if pipeline > 1:
                name = "gdr_chunk_fwd_gated_pipelined"
                st = lib().gdr_chunk_fwd_gated_pipelined(
                    ctypes.byref(shape), int(pipeline), *ins, ctypes.byref(gate), *tail,
                    _stream(aux if aux is not None else aux_stream(dev), dev))
            else:
                name = "gdr_chunk_fwd_gated"
                st = lib().gdr_chunk_fwd_gated(ctypes.byref(shape), *ins, ctypes.byref(gate),
                                               *tail)
        if st:
            raise GdrError(st, name)
        return o, hT
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam), _ptr(b), _ptr(w),
            _ptr(h0), _ptr(o), _ptr(hT), _ptr(workspace),
            ctypes.c_size_t(0 if workspace is None else workspace.numel()), _stream(stream, dev))
    with torch.cuda.device(dev):
        if pipeline > 1:
            name = "gdr_chunk_fwd_pipelined"
            st = lib().gdr_chunk_fwd_pipelined(ctypes.byref(shape), int(pipeline), *args,
                                               _stream(aux if aux is not None else aux_stream(dev),
                                                       dev))
        elif segments is None:
            name = "gdr_chunk_fwd"
            st = lib().gdr_chunk_fwd(ctypes.byref(shape), *args)
        else:
            name = "gdr_chunk_fwd_split"
            st = lib().gdr_chunk_fwd_split(ctypes.byref(shape), int(segments), *args)
    if st:
        raise GdrError(st, name)
    return o, hT


def token_fwd(q, k, v, g, beta=None, lam=None, b=None, w=None, h0=None, *, scale=None,
              flags=None, output_final_state=True, o=None, hT=None, stream=None):
    """The forward token by token (``gdr_token_fwd``): no decay factoring, so no
    range limit on the log-decay; same arguments and results as chunk_fwd."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if flags is None:
        flags = _infer_flags(g.dim() == 4, b, w, lam, beta is not None and beta.dim() == 4)
    if scale is None:
        scale = dk ** -0.5
    for name, t, want, shp in (("q", q, dt, (B, T, H, dk)), ("k", k, dt, (B, T, H, dk)),
                               ("v", v, dt, (B, T, H, dv)), ("b", b, dt, (B, T, H, dk)),
                               ("w", w, dt, (B, T, H, dv)), ("lam", lam, torch.float32, (B, T, H)),
                               ("h0", h0, torch.float32, (B, H, dk, dv))):
        _check(t, name, want, dev, shp)
    _check(g, "g", torch.float32, dev, (B, T, H, dk) if flags & DECAY_CHANNEL else (B, T, H))
    _check(beta, "beta", torch.float32, dev,
           (B, T, H, dv) if flags & BETA_CHANNEL else (B, T, H))
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=dt, device=dev)
    _check(o, "o", dt, dev, (B, T, H, dv))
    if hT is None and output_final_state:
        hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    _check(hT, "hT", torch.float32, dev, (B, H, dk, dv))
    shape = make_shape(B, T, H, dk, dv, dt, flags, scale)
    with torch.cuda.device(dev):
        st = lib().gdr_token_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(lam), _ptr(b), _ptr(w), _ptr(h0), _ptr(o),
                                 _ptr(hT), _stream(stream, dev))
    if st:
        raise GdrError(st, "gdr_token_fwd")
    return o, hT


def chunk_fwd_check(workspace, stream=None):
    """Status a chunk_fwd call left in its workspace (synchronises the stream).

    Returns None when the call completed; raises GdrError(GDR_ERR_TIMEOUT) when a
    bounded device-side wait gave up, GdrError(GDR_ERR_RANGE) when a chunk's
    summed channel log-decay was below the chunked path's limit.
    """
    if workspace is None or workspace.numel() < 256:   # no status words: nothing to check
        return None
    detail = (ctypes.c_int * 2)()
    with torch.cuda.device(workspace.device):
        st = lib().gdr_chunk_fwd_check(_ptr(workspace), _stream(stream, workspace.device), detail)
    if st == 6:
        raise GdrError(st, "gdr_chunk_fwd (sequence %d, chunk %d)" % (detail[0], detail[1]))
    if st:
        raise GdrError(st, "gdr_chunk_fwd (CTA %d, wait %d)" % (detail[0], detail[1]))
    return None


def recurrent_step(q, k, v, g, state, beta=None, lam=None, b=None, w=None, *, scale=None,
                   flags=None, o=None, stream=None):
    """One decode step (``gdr_recurrent_step``); updates ``state`` in place.

    q, k: [N, H, d_k] (or [N, 1, H, d_k]); v: [N, H, d_v]; g: [N, H] or
    [N, H, d_k]; beta / lam: [N, H]; b: [N, H, d_k]; w: [N, H, d_v];
    state: [N, H, d_k, d_v] fp32. Returns o [N, H, d_v].
    """
    N, H, dk, dv = state.shape
    dev, dt = q.device, q.dtype
    if flags is None:
        flags = _infer_flags(g.numel() == N * H * dk, b, w, lam,
                             beta is not None and beta.numel() == N * H * dv)
    if scale is None:
        scale = dk ** -0.5
    nbeta = N * H * dv if flags & BETA_CHANNEL else N * H
    for name, t, n in (("q", q, N * H * dk), ("k", k, N * H * dk), ("v", v, N * H * dv),
                       ("b", b, N * H * dk), ("w", w, N * H * dv), ("beta", beta, nbeta),
                       ("lam", lam, N * H),
                       ("g", g, N * H * dk if flags & DECAY_CHANNEL else N * H)):
        if t is not None:
            want = torch.float32 if name in ("beta", "lam", "g") else dt
            _check(t, name, want, dev)
            if t.numel() != n:
                raise ValueError("%s has %d elements, expected %d" % (name, t.numel(), n))
    _check(state, "state", torch.float32, dev)
    if o is None:
        o = torch.empty(N, H, dv, dtype=dt, device=dev)
    _check(o, "o", dt, dev)
    shape = make_shape(N, 1, H, dk, dv, dt, flags, scale)
    with torch.cuda.device(dev):
        st = lib().gdr_recurrent_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      _ptr(beta), _ptr(lam), _ptr(b), _ptr(w), _ptr(state),
                                      _ptr(o), _stream(stream, dev))
    if st:
        raise GdrError(st, "gdr_recurrent_step")
    return o


def gate_cumsum(g, chunk=CHUNK, out=None, stream=None):
    """Chunk-local inclusive cumsum of g ([B, T, H] or [B, T, H, d_k], fp32)."""
    B, T = g.shape[0], g.shape[1]
    X = g.numel() // max(B * T, 1)
    _check(g, "g", torch.float32, g.device)
    if out is None:
        out = torch.empty_like(g)
    _check(out, "out", torch.float32, g.device, tuple(g.shape))
    with torch.cuda.device(g.device):
        st = lib().gdr_gate_cumsum(B, T, X, chunk, _ptr(g), _ptr(out), _stream(stream, g.device))
    if st:
        raise GdrError(st, "gdr_gate_cumsum")
    return out


def rmsnorm_gate(o, z, weight, eps=1e-6, *, out=None, stream=None):
    """Output epilogue (``gdr_rmsnorm_gate``): RMSNorm of o over its last axis
    (d_v), times ``weight``, times silu(z).

    o, z: [..., d_v] bf16 or fp32 (one dtype, contiguous); weight: [d_v] fp32.
    ``out`` may be o or z itself (in place); by default a new tensor.
    """
    dv = o.shape[-1]
    dev, dt = o.device, o.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("o and z must be bf16 or fp32")
    _check(o, "o", dt, dev)
    _check(z, "z", dt, dev, tuple(o.shape))
    _check(weight, "weight", torch.float32, dev, (dv,))
    if out is None:
        out = torch.empty_like(o)
    _check(out, "out", dt, dev, tuple(o.shape))
    rows = o.numel() // dv if dv else 0
    with torch.cuda.device(dev):
        st = lib().gdr_rmsnorm_gate(rows, dv, GDR_BF16 if dt == torch.bfloat16 else GDR_F32,
                                    _ptr(o), _ptr(z), _ptr(weight), ctypes.c_float(eps),
                                    _ptr(out), _stream(stream, dev))
    if st:
        raise GdrError(st, "gdr_rmsnorm_gate")
    return out


def chunk_bwd_workspace_bytes(shape):
    n = ctypes.c_size_t(0)
    st = lib().gdr_chunk_bwd_workspace(ctypes.byref(shape), ctypes.byref(n))
    if st:
        raise GdrError(st, "gdr_chunk_bwd_workspace")
    return n.value


def chunk_bwd_check(workspace, stream=None):
    """Status a chunk_bwd call left in its workspace (synchronises the stream):
    None, or GdrError(GDR_ERR_RANGE) when a chunk's log-decay left the
    backward's range (the gradients are then not to be used)."""
    detail = (ctypes.c_int * 2)()
    with torch.cuda.device(workspace.device):
        st = lib().gdr_chunk_bwd_check(_ptr(workspace), _stream(stream, workspace.device), detail)
    if st == 6:
        raise GdrError(st, "gdr_chunk_bwd (sequence %d, chunk %d)" % (detail[0], detail[1]))
    if st:
        raise GdrError(st, "gdr_chunk_bwd_check")
    return None


def _bwd(token, q, k, v, g, dO, beta=None, lam=None, b=None, w=None, h0=None, dhT=None, *,
         scale=None, flags=None, workspace=None, stream=None, check=False):
    """Shared body of chunk_bwd and token_bwd."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if flags is None:
        flags = _infer_flags(g.dim() == 4, b, w, lam, beta is not None and beta.dim() == 4)
    if scale is None:
        scale = dk ** -0.5
    _check(dO, "dO", dt, dev, (B, T, H, dv))
    _check(dhT, "dhT", torch.float32, dev, (B, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"q": torch.empty(B, T, H, dk, **f32), "k": torch.empty(B, T, H, dk, **f32),
           "v": torch.empty(B, T, H, dv, **f32), "g": torch.empty(tuple(g.shape), **f32),
           "beta": None if beta is None else torch.empty(tuple(beta.shape), **f32),
           "lam": None if lam is None else torch.empty(B, T, H, **f32),
           "b": None if b is None else torch.empty(B, T, H, dk, **f32),
           "w": None if w is None else torch.empty(B, T, H, dv, **f32),
           "h0": torch.empty(B, H, dk, dv, **f32)}
    shape = make_shape(B, T, H, dk, dv, dt, flags, scale)
    if workspace is None:
        nbytes = (token_bwd_workspace_bytes if token else chunk_bwd_workspace_bytes)(shape)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        fn = lib().gdr_token_bwd if token else lib().gdr_chunk_bwd
        st = fn(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(lam), _ptr(b), _ptr(w), _ptr(h0), _ptr(dO),
                                 _ptr(dhT), *(_ptr(out[n]) for n in
                                              ("q", "k", "v", "g", "beta", "lam", "b", "w",
                                               "h0")),
                                 _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                 _stream(stream, dev))
    if st:
        raise GdrError(st, "gdr_token_bwd" if token else "gdr_chunk_bwd")
    if check:
        chunk_bwd_check(workspace, stream)
    return out


def chunk_bwd(q, k, v, g, dO, beta=None, lam=None, b=None, w=None, h0=None, dhT=None, *,
              scale=None, flags=None, workspace=None, stream=None, check=False):
    """Gradients of <dO, o> + <dhT, hT> for ``chunk_fwd`` on the same inputs
    (``gdr_chunk_bwd``). Returns a dict of fp32 tensors: q, k, v, g, and beta,
    lam, b, w, h0 where they apply (None otherwise). With check=True the call
    synchronises and raises GdrError(GDR_ERR_RANGE) for inputs past the
    backward's decay range (chunk_bwd_check)."""
    return _bwd(False, q, k, v, g, dO, beta, lam, b, w, h0, dhT, scale=scale, flags=flags,
                workspace=workspace, stream=stream, check=check)


def token_bwd_workspace_bytes(shape):
    n = ctypes.c_size_t(0)
    st = lib().gdr_token_bwd_workspace(ctypes.byref(shape), ctypes.byref(n))
    if st:
        raise GdrError(st, "gdr_token_bwd_workspace")
    return n.value


def token_bwd(q, k, v, g, dO, beta=None, lam=None, b=None, w=None, h0=None, dhT=None, *,
              scale=None, flags=None, workspace=None, stream=None):
    """chunk_bwd's gradients walked token by token (``gdr_token_bwd``): no decay
    range limit, for inputs chunk_bwd reports as GDR_ERR_RANGE. Same arguments
    and result."""
    return _bwd(True, q, k, v, g, dO, beta, lam, b, w, h0, dhT, scale=scale, flags=flags,
                workspace=workspace, stream=stream)
