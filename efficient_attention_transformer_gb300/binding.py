"""ctypes binding of libflashgau (see include/flash_gau.h).

Argument marshalling only: tensors are checked for device, dtype and
contiguity and their data pointers handed to the C entry points; every step
of the computation runs in the library's CUDA kernels.  Loading fails loudly
when the library has not been built.
"""

import ctypes
import os

import torch

from .build import LIB as _LIB_PATH

FP32 = 0
BF16 = 1

OK = 0
EINVAL = -1
ENOTSUP = -2
EWORKSPACE = -3
ECUDA = -4
EDEVICE = -5
ETIMEOUT = -6

NORM_NONE = 0
NORM_LAYER = 1
NORM_SCALE = 2

# Every function the header declares; the library must export all of them.
EXPORTED = (
    "flash_gau_workspace_layout_query",
    "flash_gau_workspace_bytes",
    "flash_gau_forward",
    "flash_gau_forward_timed",
    "flash_gau_num_stages",
    "flash_gau_stage_name",
    "flash_gau_workspace_status",
    "flash_gau_strerror",
    "flash_gau_version",
    "flash_gau_forward_noalloc",
    "flash_gau_block_forward",
    "flash_gau_rope_toeplitz_bias",
    "flash_gau_backward_workspace_bytes",
    "flash_gau_backward",
    "flash_gau_decode_state_bytes",
    "flash_gau_decode_step",
    "flash_gau_forward_segmented",
    "flash_gau_forward_host_workspace_bytes",
    "flash_gau_forward_host",
    "flash_gau_selftest_bounded_wait",
)

# Capacity of the static scratch behind flash_gau_forward_noalloc.
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class Segments(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("average", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [
        ("W_uvz", ctypes.c_void_p),
        ("W_o", ctypes.c_void_p),
        ("gamma", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("relpos", ctypes.c_void_p),
        ("d", ctypes.c_int),
        ("e", ctypes.c_int),
        ("s", ctypes.c_int),
        ("lin_scale", ctypes.c_float),
        ("local_scale", ctypes.c_float),
    ]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("total_bytes", "status", "U", "V", "heads", "state", "prefix", "gated",
                 "bias", "xn", "rope")]


class Block(ctypes.Structure):
    """flash_gau_block: the flash_block options (norm, RoPE, residual)."""
    _fields_ = [
        ("norm", ctypes.c_int),
        ("norm_g", ctypes.c_void_p),
        ("norm_b", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
        ("rope", ctypes.c_int),
        ("rope_base", ctypes.c_float),
        ("pos_offset", ctypes.c_int),
        ("residual", ctypes.c_int),
    ]


class FlashGauError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("flash_gau status %d: %s" % (status, msg))
        self.status = status


_lib = None


def lib():
    """The loaded library (loaded on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "libflashgau.so is not built (expected at %s); call "
                "efficient_attention_transformer_gb300.build.build()" % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        i, p, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.flash_gau_workspace_layout_query.argtypes = [i, i, i, i, i, i, i, i,
                                                       ctypes.POINTER(WorkspaceLayout)]
        L.flash_gau_workspace_layout_query.restype = i
        L.flash_gau_workspace_bytes.argtypes = [i, i, i, ctypes.POINTER(Weights), i, i]
        L.flash_gau_workspace_bytes.restype = sz
        L.flash_gau_forward.argtypes = [p, ctypes.POINTER(Weights), i, i, i, i, i, p, p, sz, p]
        L.flash_gau_forward.restype = i
        L.flash_gau_forward_timed.argtypes = [p, ctypes.POINTER(Weights), i, i, i, i, i, p, p,
                                              sz, p, ctypes.POINTER(p), i]
        L.flash_gau_forward_timed.restype = i
        L.flash_gau_num_stages.argtypes = [i, i]
        L.flash_gau_num_stages.restype = i
        L.flash_gau_stage_name.argtypes = [i, i, i]
        L.flash_gau_stage_name.restype = ctypes.c_char_p
        L.flash_gau_workspace_status.argtypes = [p, p]
        L.flash_gau_workspace_status.restype = i
        L.flash_gau_strerror.argtypes = [i]
        L.flash_gau_strerror.restype = ctypes.c_char_p
        L.flash_gau_version.argtypes = []
        L.flash_gau_version.restype = i
        L.flash_gau_forward_noalloc.argtypes = [p, ctypes.POINTER(Weights), i, i, i, i, i, p, p]
        L.flash_gau_forward_noalloc.restype = i
        L.flash_gau_block_forward.argtypes = [p, ctypes.POINTER(Weights), ctypes.POINTER(Block),
                                              i, i, i, i, i, p, p, sz, p]
        L.flash_gau_block_forward.restype = i
        L.flash_gau_forward_segmented.argtypes = [p, ctypes.POINTER(Weights),
                                                  ctypes.POINTER(Segments), i, i, i, i, i, p,
                                                  p, sz, p]
        L.flash_gau_forward_segmented.restype = i
        L.flash_gau_forward_host_workspace_bytes.argtypes = [i, i, i, ctypes.POINTER(Weights),
                                                             i, i]
        L.flash_gau_forward_host_workspace_bytes.restype = sz
        L.flash_gau_forward_host.argtypes = [p, ctypes.POINTER(Weights), i, i, i, i, i, p, p,
                                             sz, p]
        L.flash_gau_forward_host.restype = i
        L.flash_gau_selftest_bounded_wait.argtypes = [i, p, p]
        L.flash_gau_selftest_bounded_wait.restype = i
        L.flash_gau_rope_toeplitz_bias.argtypes = [p, p, i, i, ctypes.c_float, p, p]
        L.flash_gau_rope_toeplitz_bias.restype = i
        L.flash_gau_backward_workspace_bytes.argtypes = [i, i, i, ctypes.POINTER(Weights), i, i]
        L.flash_gau_backward_workspace_bytes.restype = sz
        L.flash_gau_backward.argtypes = [p, p, ctypes.POINTER(Weights), i, i, i, i, i,
                                         ctypes.POINTER(Grads), p, sz, p]
        L.flash_gau_backward.restype = i
        L.flash_gau_decode_state_bytes.argtypes = [i, i, ctypes.POINTER(Weights), i]
        L.flash_gau_decode_state_bytes.restype = sz
        L.flash_gau_decode_step.argtypes = [p, ctypes.POINTER(Weights), i, i, i, p, sz, p, p]
        L.flash_gau_decode_step.restype = i
        _lib = L
    return _lib


def strerror(status):
    return lib().flash_gau_strerror(status).decode()


def _check(status):
    if status != OK:
        raise FlashGauError(status, strerror(status))


def dtype_code(t):
    if t == torch.float32:
        return FP32
    if t == torch.bfloat16:
        return BF16
    raise TypeError("io dtype must be float32 or bfloat16, got %s" % (t,))


def workspace_layout(B, T, C, d, e, s, causal, dtype):
    """Byte offsets of the intermediates, as a dict."""
    L = WorkspaceLayout()
    _check(lib().flash_gau_workspace_layout_query(B, T, C, d, e, s, int(bool(causal)),
                                                  dtype, ctypes.byref(L)))
    return {n: getattr(L, n) for n, _ in WorkspaceLayout._fields_}


def num_stages(dtype, causal):
    return lib().flash_gau_num_stages(dtype, int(bool(causal)))


def stage_names(dtype, causal):
    return [lib().flash_gau_stage_name(dtype, int(bool(causal)), k).decode()
            for k in range(num_stages(dtype, causal))]


def _dev_ptr(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


class Grads(ctypes.Structure):
    _fields_ = [("dX", ctypes.c_void_p), ("dW_uvz", ctypes.c_void_p), ("dW_o", ctypes.c_void_p),
                ("dgamma", ctypes.c_void_p), ("dbeta", ctypes.c_void_p),
                ("drelpos", ctypes.c_void_p)]


class GauWeights:
    """Device-resident layer parameters in the layout the library expects."""

    def __init__(self, W_uvz, W_o, gamma, beta, relpos, d, e, s, lin_scale=1.0,
                 local_scale=1.0):
        self.W_uvz, self.W_o = W_uvz, W_o
        self.gamma, self.beta, self.relpos = gamma, beta, relpos
        self.d, self.e, self.s = int(d), int(e), int(s)
        self.lin_scale, self.local_scale = float(lin_scale), float(local_scale)
        self.dtype = dtype_code(W_uvz.dtype)
        f32 = torch.float32
        self.c = Weights(_dev_ptr(W_uvz, "W_uvz", W_uvz.dtype), _dev_ptr(W_o, "W_o", W_uvz.dtype),
                         _dev_ptr(gamma, "gamma", f32), _dev_ptr(beta, "beta", f32),
                         _dev_ptr(relpos, "relpos", f32), self.d, self.e, self.s,
                         self.lin_scale, self.local_scale)
        if tuple(W_uvz.shape) != (d, 2 * e + s) or tuple(W_o.shape) != (e, d):
            raise ValueError("weight shapes do not match d, e, s")
        if tuple(gamma.shape) != (4, s) or tuple(beta.shape) != (4, s):
            raise ValueError("gamma and beta must be [4, s]")

    def workspace_bytes(self, B, T, C, causal):
        n = lib().flash_gau_workspace_bytes(B, T, C, ctypes.byref(self.c), int(bool(causal)),
                                            self.dtype)
        if n == 0:
            raise FlashGauError(EINVAL, "invalid or unsupported problem")
        return n

    def new_workspace(self, B, T, C, causal, device=None):
        n = self.workspace_bytes(B, T, C, causal)
        return torch.zeros(n, dtype=torch.uint8, device=device or self.W_uvz.device)


def forward(X, weights, C, causal, out=None, workspace=None, stream=None,
            stage_events=None):
    """O = FLASH-GAU(X) through flash_gau_forward (or _timed when
    stage_events, a list of torch.cuda.Event, is given).  X: [B, T, d]."""
    if X.dim() != 3:
        raise ValueError("X must be [B, T, d]")
    B, T, d = X.shape
    if d != weights.d:
        raise ValueError("X width does not match the weights")
    if X.dtype != weights.W_uvz.dtype:
        raise ValueError("X and weights must share the io dtype")
    if weights.relpos.numel() != 2 * C - 1:
        raise ValueError("relpos must hold 2C-1 values")
    if out is None:
        out = torch.empty_like(X)
    if workspace is None:
        workspace = weights.new_workspace(B, T, C, causal, X.device)
    if stream is None:
        stream = torch.cuda.current_stream(X.device)
    sp = stream.cuda_stream
    args = (_dev_ptr(X, "X", X.dtype), ctypes.byref(weights.c), B, T, C, int(bool(causal)),
            weights.dtype, _dev_ptr(out, "out", X.dtype), _dev_ptr(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), sp)
    if stage_events:
        for ev in stage_events:  # torch creates the CUDA event on first record
            if not ev.cuda_event:
                ev.record(stream)
        arr = (ctypes.c_void_p * len(stage_events))(*[ev.cuda_event for ev in stage_events])
        st = lib().flash_gau_forward_timed(*args, arr, len(stage_events))
    else:
        st = lib().flash_gau_forward(*args)
    _check(st)
    return out


def forward_segmented(X, weights, C, causal, segment_ids=None, average=False, out=None,
                      workspace=None, stream=None):
    """O = FLASH-GAU(X) with a chunk mask on the global term, through
    flash_gau_forward_segmented.  segment_ids: int32 CUDA tensor [B, T / C]
    (one id per chunk; a change of id starts a segment) or None; average:
    the mean of the visible chunk states instead of their sum."""
    if X.dim() != 3:
        raise ValueError("X must be [B, T, d]")
    B, T, d = X.shape
    if d != weights.d or X.dtype != weights.W_uvz.dtype:
        raise ValueError("X does not match the weights")
    ids = None
    if segment_ids is not None:
        if T % C != 0 or tuple(segment_ids.shape) != (B, T // C):
            raise ValueError("segment_ids must be [B, T / C]")
        ids = _dev_ptr(segment_ids, "segment_ids", torch.int32)
    seg = Segments(ids, int(bool(average)))
    if out is None:
        out = torch.empty_like(X)
    if workspace is None:
        workspace = weights.new_workspace(B, T, C, causal, X.device)
    if stream is None:
        stream = torch.cuda.current_stream(X.device)
    _check(lib().flash_gau_forward_segmented(
        _dev_ptr(X, "X", X.dtype), ctypes.byref(weights.c), ctypes.byref(seg), B, T, C,
        int(bool(causal)), weights.dtype, _dev_ptr(out, "out", X.dtype),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        stream.cuda_stream))
    return out


def forward_host(X, weights, C, causal, out=None, workspace=None, stream=None):
    """O = FLASH-GAU(X) on host tensors through flash_gau_forward_host: X is
    a CPU tensor [B, T, d] (pinned for overlapped copies), the result goes to
    `out` (a CPU tensor like X; allocated pinned when None).  The call
    returns once the work is queued on `stream`; synchronise it before
    reading `out`."""
    if X.dim() != 3 or X.is_cuda:
        raise ValueError("X must be a CPU tensor [B, T, d]")
    if not X.is_contiguous():
        raise ValueError("X must be contiguous")
    B, T, d = X.shape
    if d != weights.d or X.dtype != weights.W_uvz.dtype:
        raise ValueError("X does not match the weights")
    if out is None:
        out = torch.empty_like(X).pin_memory()
    if out.is_cuda or out.shape != X.shape or out.dtype != X.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU tensor like X")
    dev = weights.W_uvz.device
    if workspace is None:
        n = lib().flash_gau_forward_host_workspace_bytes(B, T, C, ctypes.byref(weights.c),
                                                         int(bool(causal)), weights.dtype)
        if n == 0:
            raise FlashGauError(EINVAL, "invalid or unsupported problem")
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    _check(lib().flash_gau_forward_host(
        X.data_ptr(), ctypes.byref(weights.c), B, T, C, int(bool(causal)), weights.dtype,
        out.data_ptr(), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), stream.cuda_stream))
    return out


def forward_noalloc(X, weights, C, causal, out=None, stream=None):
    """O = FLASH-GAU(X) through flash_gau_forward_noalloc: no workspace, the
    intermediates live in the library's static 32 MiB device scratch (shared
    by every call on the device; calls must not overlap on the GPU)."""
    if X.dim() != 3:
        raise ValueError("X must be [B, T, d]")
    B, T, d = X.shape
    if d != weights.d or X.dtype != weights.W_uvz.dtype:
        raise ValueError("X does not match the weights")
    if out is None:
        out = torch.empty_like(X)
    # the library picks the scratch of the current device: make it X's
    with torch.cuda.device(X.device):
        if stream is None:
            stream = torch.cuda.current_stream(X.device)
        _check(lib().flash_gau_forward_noalloc(
            _dev_ptr(X, "X", X.dtype), ctypes.byref(weights.c), B, T, C, int(bool(causal)),
            weights.dtype, _dev_ptr(out, "out", X.dtype), stream.cuda_stream))
    return out


def block_forward(X, weights, C, causal, norm=NORM_LAYER, norm_g=None, norm_b=None,
                  norm_eps=1e-5, rope=True, rope_base=10000.0, pos_offset=0, residual=True,
                  out=None, workspace=None, stream=None):
    """Y = X + layer(norm(X)) with RoPE on the heads, through
    flash_gau_block_forward.  norm_g / norm_b: fp32 CUDA tensors ([d] for
    LayerNorm, [1] for ScaleNorm's g; norm_b may be None)."""
    if X.dim() != 3:
        raise ValueError("X must be [B, T, d]")
    B, T, d = X.shape
    if d != weights.d or X.dtype != weights.W_uvz.dtype:
        raise ValueError("X does not match the weights")
    f32 = torch.float32
    blk = Block(int(norm),
                _dev_ptr(norm_g, "norm_g", f32) if norm_g is not None else None,
                _dev_ptr(norm_b, "norm_b", f32) if norm_b is not None else None,
                float(norm_eps), int(bool(rope)), float(rope_base), int(pos_offset),
                int(bool(residual)))
    if out is None:
        out = torch.empty_like(X)
    if workspace is None:
        workspace = weights.new_workspace(B, T, C, causal, X.device)
    if stream is None:
        stream = torch.cuda.current_stream(X.device)
    _check(lib().flash_gau_block_forward(
        _dev_ptr(X, "X", X.dtype), ctypes.byref(weights.c), ctypes.byref(blk), B, T, C,
        int(bool(causal)), weights.dtype, _dev_ptr(out, "out", X.dtype),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        stream.cuda_stream))
    return out


def workspace_status(workspace, stream=None):
    """Synchronises and returns (and clears) the kernels' status word."""
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return lib().flash_gau_workspace_status(_dev_ptr(workspace, "workspace"), stream.cuda_stream)


def rope_toeplitz_bias(a, b, C, rope_base=10000.0, out=None, stream=None):
    """The layer's relative-position table [2C-1] (fp32, device) of the RoPE
    bias construction from the learned vectors a, b ([m] fp32 CUDA tensors),
    through flash_gau_rope_toeplitz_bias."""
    f32 = torch.float32
    if a.shape != b.shape or a.dim() != 1:
        raise ValueError("a and b must be vectors of the same length")
    if out is None:
        out = torch.empty(2 * C - 1, dtype=f32, device=a.device)
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    _check(lib().flash_gau_rope_toeplitz_bias(
        _dev_ptr(a, "a", f32), _dev_ptr(b, "b", f32), a.numel(), C, float(rope_base),
        _dev_ptr(out, "out", f32), stream.cuda_stream))
    return out


def backward(X, dO, weights, C, causal, workspace=None, stream=None):
    """Gradients of sum(dO * O) through flash_gau_backward: a dict with dX
    (io type) and dW_uvz, dW_o, dgamma, dbeta, drelpos (fp32), on X's
    device."""
    if X.dim() != 3 or dO.shape != X.shape:
        raise ValueError("X and dO must be [B, T, d]")
    B, T, d = X.shape
    if d != weights.d or X.dtype != weights.W_uvz.dtype or dO.dtype != X.dtype:
        raise ValueError("X, dO and the weights must agree")
    f32, dev = torch.float32, X.device
    e, s = weights.e, weights.s
    out = dict(dX=torch.empty_like(X),
               dW_uvz=torch.empty(d, 2 * e + s, dtype=f32, device=dev),
               dW_o=torch.empty(e, d, dtype=f32, device=dev),
               dgamma=torch.empty(4, s, dtype=f32, device=dev),
               dbeta=torch.empty(4, s, dtype=f32, device=dev),
               drelpos=torch.empty(2 * C - 1, dtype=f32, device=dev))
    g = Grads(*(_dev_ptr(out[k], k) for k in ("dX", "dW_uvz", "dW_o", "dgamma", "dbeta",
                                             "drelpos")))
    n = lib().flash_gau_backward_workspace_bytes(B, T, C, ctypes.byref(weights.c),
                                                 int(bool(causal)), weights.dtype)
    if n == 0:
        raise FlashGauError(EINVAL, "invalid or unsupported problem")
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    _check(lib().flash_gau_backward(
        _dev_ptr(X, "X", X.dtype), _dev_ptr(dO, "dO", X.dtype), ctypes.byref(weights.c), B, T, C,
        int(bool(causal)), weights.dtype, ctypes.byref(g), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), stream.cuda_stream))
    return out


class Decoder:
    """B sequences decoded one token per call through flash_gau_decode_step;
    the state lives on the weights' device and starts all sequences at
    position 0."""

    def __init__(self, weights, B, C):
        self.weights, self.B, self.C = weights, int(B), int(C)
        n = lib().flash_gau_decode_state_bytes(self.B, self.C, ctypes.byref(weights.c),
                                               weights.dtype)
        if n == 0:
            raise FlashGauError(EINVAL, "invalid or unsupported decode problem")
        self.state = torch.zeros(n, dtype=torch.uint8, device=weights.W_uvz.device)

    def reset(self):
        self.state.zero_()

    def step(self, x, out=None, stream=None):
        """x: [B, d] in the io type; returns the [B, d] outputs."""
        if tuple(x.shape) != (self.B, self.weights.d) or x.dtype != self.weights.W_uvz.dtype:
            raise ValueError("x must be [B, d] in the weights' type")
        if out is None:
            out = torch.empty_like(x)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        _check(lib().flash_gau_decode_step(
            _dev_ptr(x, "x", x.dtype), ctypes.byref(self.weights.c), self.B, self.C,
            self.weights.dtype, _dev_ptr(self.state, "state"), self.state.numel(),
            _dev_ptr(out, "out", x.dtype), stream.cuda_stream))
        return out
