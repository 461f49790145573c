"""Python binding of the GB300 Muon optimizer-step library (``libmuon_gb300.so``).

Argument marshalling only: every step of the Muon step runs in the CUDA
kernels of the library, which is loaded with ctypes.  torch supplies device
memory and the stream handle.  There is no CPU or eager fallback: if the
library is not built, every call raises.

The functions mirror the C ABI in ``include/muon.h``:

    muon_ns5_batched(mats, steps=5, coeffs=None, stream=None)
    muon_step(W, G, M, lr, mu, wd, stream=None)
    muon_step_ex(W, G, M, lr, mu, wd, *, steps, coeffs, eps, nesterov, workspace, stream)
    muon_workspace_bytes(shapes)
    muon_device_status(stream=None)
    muon_release_workspace()
    muon_profile_enable(on), muon_profile_read()

The method: the per-matrix Muon step over whole matrices held on one rank
("How PyTorch Scaled a Near-1T MoE on Europe's Public Supercomputer", section
"Three optimizations that changed the economics", FlexShard bullet).
"""
import ctypes
import os

import torch

__all__ = [
    "MuonError", "lib", "LIB_PATH", "EXPORTS", "DEFAULT_COEFFS",
    "muon_ns5_batched", "muon_step", "muon_step_ex", "muon_workspace_bytes",
    "muon_device_status", "muon_release_workspace", "muon_profile_enable",
    "muon_profile_read", "muon_status_string", "MuonStepBatch", "muon_ns5_batched_static",
    "MUON_STATIC_SCRATCH_BYTES", "muon_step_host", "muon_ns_batched_ex", "muon_adamw_step",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmuon_gb300.so")
DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)

# every entry point declared in include/muon.h
EXPORTS = (
    "muon_ns5_batched", "muon_step", "muon_step_opts_init", "muon_step_ex",
    "muon_workspace_bytes", "muon_status_string", "muon_last_error",
    "muon_device_status", "muon_release_workspace", "muon_profile_enable",
    "muon_profile_read", "muon_ns5_batched_static", "muon_step_host", "muon_ns_batched_ex",
    "muon_adamw_step",
)

MUON_STATIC_SCRATCH_BYTES = 64 << 20

MUON_BF16, MUON_F32 = 0, 1


class MuonError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"status {status}: {detail}")


class _Opts(ctypes.Structure):
    _fields_ = [("w_dtype", ctypes.c_int), ("g_dtype", ctypes.c_int), ("steps", ctypes.c_int),
                ("coeffs", ctypes.POINTER(ctypes.c_float)), ("eps", ctypes.c_float),
                ("nesterov", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("o_out", ctypes.POINTER(ctypes.c_void_p)),
                ("coeffs_per_step", ctypes.c_int), ("g_count", ctypes.c_int), ("ns_fp8_gram", ctypes.c_int)]


class _KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


_lib = None


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m muon_newton_schulz_step_gb300.build` "
            "(nvcc, sm_103a). There is no fallback implementation.")
    L = ctypes.CDLL(LIB_PATH)
    vp, ip, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    L.muon_ns5_batched.argtypes = [vpp, ip, ip, ctypes.c_int, ctypes.c_int, fp, vp]
    L.muon_ns5_batched.restype = ctypes.c_int
    L.muon_ns_batched_ex.argtypes = [vpp, ip, ip, ctypes.c_int, ctypes.c_int, fp, ctypes.c_int, vp]
    L.muon_ns_batched_ex.restype = ctypes.c_int
    L.muon_ns5_batched_static.argtypes = [vpp, ip, ip, ctypes.c_int, ctypes.c_int, fp, vp]
    L.muon_ns5_batched_static.restype = ctypes.c_int
    L.muon_step.argtypes = [vpp, vpp, vpp, ip, ip, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                            ctypes.c_float, vp]
    L.muon_step.restype = ctypes.c_int
    L.muon_step_opts_init.argtypes = [ctypes.POINTER(_Opts)]
    L.muon_step_opts_init.restype = None
    L.muon_step_ex.argtypes = [vpp, vpp, vpp, ip, ip, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                               ctypes.c_float, ctypes.POINTER(_Opts), vp]
    L.muon_step_ex.restype = ctypes.c_int
    L.muon_step_host.argtypes = [vpp, vpp, vpp, ip, ip, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                 ctypes.c_float, ctypes.POINTER(_Opts), vp]
    L.muon_step_host.restype = ctypes.c_int
    L.muon_adamw_step.argtypes = [vpp, vpp, vpp, vpp, ctypes.POINTER(ctypes.c_longlong), ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  ctypes.c_float, ctypes.c_float, ctypes.c_int, vp]
    L.muon_adamw_step.restype = ctypes.c_int
    L.muon_workspace_bytes.argtypes = [ip, ip, ctypes.c_int]
    L.muon_workspace_bytes.restype = ctypes.c_size_t
    L.muon_status_string.argtypes = [ctypes.c_int]
    L.muon_status_string.restype = ctypes.c_char_p
    L.muon_last_error.argtypes = []
    L.muon_last_error.restype = ctypes.c_char_p
    L.muon_device_status.argtypes = [vp, ip]
    L.muon_device_status.restype = ctypes.c_int
    L.muon_release_workspace.argtypes = []
    L.muon_release_workspace.restype = None
    L.muon_profile_enable.argtypes = [ctypes.c_int]
    L.muon_profile_enable.restype = ctypes.c_int
    L.muon_profile_read.argtypes = [ctypes.POINTER(_KernelStat), ctypes.c_int, ip]
    L.muon_profile_read.restype = ctypes.c_int
    _lib = L
    return L


def muon_status_string(status: int) -> str:
    return lib().muon_status_string(int(status)).decode()


def _check(rc: int):
    if rc != 0:
        raise MuonError(rc, lib().muon_last_error().decode())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr_array(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _dims(tensors):
    n = len(tensors)
    rows = (ctypes.c_int * n)(*[int(t.shape[0]) for t in tensors])
    cols = (ctypes.c_int * n)(*[int(t.shape[1]) for t in tensors])
    return rows, cols


def _check_mats(name, tensors, dtypes, stacked=False):
    """Every tensor a contiguous CUDA tensor on the current device, 2-D (or
    3-D where ``stacked``), of one of ``dtypes``."""
    device = None
    for i, t in enumerate(tensors):
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name}[{i}] must be a tensor")
        ok_dim = t.dim() in (2, 3) if stacked else t.dim() == 2
        if not ok_dim or not t.is_cuda:
            raise ValueError(f"{name}[{i}] must be a {'2-D or 3-D' if stacked else '2-D'} CUDA tensor")
        device = _check_device(f"{name}[{i}]", t, device)
        if not t.is_contiguous():
            raise ValueError(f"{name}[{i}] must be contiguous")
        if t.dtype not in dtypes:
            raise ValueError(f"{name}[{i}] has dtype {t.dtype}; expected one of {dtypes}")


def _check_device(what, t, device=None):
    """``t`` must live on the current CUDA device (the library launches there);
    returns that device's index for the next call."""
    if device is None:
        device = torch.cuda.current_device()
    if t.get_device() != device:
        raise ValueError(f"{what} is on cuda:{t.get_device()}; the current device is cuda:{device}")
    return device


def _check_step_shapes(W, G, M, stacked_g):
    """W[i] is 2-D, M[i] has W[i]'s shape and G[i] is W[i]'s shape (or K x that
    shape where ``stacked_g``).  The library reads and writes rows[i] x cols[i]
    elements through each pointer, so a smaller G or M would be overrun."""
    if not (len(W) == len(G) == len(M)):
        raise ValueError("W, G and M must have the same length")
    for i, (w, g, m) in enumerate(zip(W, G, M)):
        for name, t in (("W", w), ("G", g), ("M", m)):
            if not isinstance(t, torch.Tensor):
                raise ValueError(f"{name}[{i}] must be a tensor")
        if w.dim() != 2:
            raise ValueError(f"W[{i}] must be 2-D")
        if tuple(m.shape) != tuple(w.shape):
            raise ValueError(f"M[{i}] has shape {tuple(m.shape)}; W[{i}] has {tuple(w.shape)}")
        if g.dim() not in ((2, 3) if stacked_g else (2,)) or tuple(g.shape[-2:]) != tuple(w.shape):
            raise ValueError(f"G[{i}] has shape {tuple(g.shape)}; expected W[{i}]'s {tuple(w.shape)}"
                             + (" (optionally with a leading stack dimension)" if stacked_g else ""))


def _coeff_array(coeffs):
    if coeffs is None:
        return None
    if len(coeffs) != 3:
        raise ValueError("coeffs must be (a, b, c)")
    return (ctypes.c_float * 3)(*[float(c) for c in coeffs])


def _schedule(coeffs, steps):
    """(array, per_step): one (a, b, c) triple, or a sequence of `steps` triples."""
    if coeffs is None:
        return None, 0
    if len(coeffs) > 0 and hasattr(coeffs[0], "__len__"):
        if len(coeffs) != steps or any(len(t) != 3 for t in coeffs):
            raise ValueError("a coefficient schedule needs one (a, b, c) triple per step")
        flat = [float(v) for t in coeffs for v in t]
        return (ctypes.c_float * max(1, len(flat)))(*flat), 1
    return _coeff_array(coeffs), 0


def muon_ns_batched_ex(mats, steps: int = 5, coeffs=None, stream=None) -> None:
    """muon_ns5_batched where ``coeffs`` may be one (a, b, c) triple or a
    schedule of ``steps`` triples (one per iteration)."""
    mats = list(mats)
    _check_mats("mats", mats, (torch.bfloat16,))
    rows, cols = _dims(mats)
    arr, per_step = _schedule(coeffs, int(steps))
    _check(lib().muon_ns_batched_ex(_ptr_array(mats), rows, cols, len(mats), int(steps), arr, per_step,
                                    _stream_handle(stream)))


def muon_ns5_batched(mats, steps: int = 5, coeffs=None, stream=None) -> None:
    """In-place normalise + Newton-Schulz of a list of bf16 CUDA matrices."""
    mats = list(mats)
    _check_mats("mats", mats, (torch.bfloat16,))
    rows, cols = _dims(mats)
    _check(lib().muon_ns5_batched(_ptr_array(mats), rows, cols, len(mats), int(steps),
                                  _coeff_array(coeffs), _stream_handle(stream)))


def muon_ns5_batched_static(mats, steps: int = 5, coeffs=None, stream=None) -> None:
    """muon_ns5_batched without any device allocation: the library's scratch is a
    fixed MUON_STATIC_SCRATCH_BYTES device array (for callers that cannot call
    cudaMalloc).  Batches needing more scratch raise MuonError; calls that
    overlap on the GPU race on the shared array."""
    mats = list(mats)
    _check_mats("mats", mats, (torch.bfloat16,))
    rows, cols = _dims(mats)
    _check(lib().muon_ns5_batched_static(_ptr_array(mats), rows, cols, len(mats), int(steps),
                                         _coeff_array(coeffs), _stream_handle(stream)))


def _dtype_code(t):
    return MUON_F32 if t.dtype == torch.float32 else MUON_BF16


def muon_step(W, G, M, lr: float, mu: float, wd: float, stream=None) -> None:
    """Muon step with bf16 W and G, fp32 M, defaults for everything else."""
    W, G, M = list(W), list(G), list(M)
    _check_step_shapes(W, G, M, stacked_g=False)
    _check_mats("W", W, (torch.bfloat16,))
    _check_mats("G", G, (torch.bfloat16,))
    _check_mats("M", M, (torch.float32,))
    rows, cols = _dims(W)
    _check(lib().muon_step(_ptr_array(W), _ptr_array(G), _ptr_array(M), rows, cols, len(W),
                           float(lr), float(mu), float(wd), _stream_handle(stream)))


def _g_count(W, G):
    """Gradients per matrix: G[i] is rows x cols, or K x rows x cols (K stacked
    gradients summed in fp32 by the library); every G[i] must use the same K."""
    ks = {1 if g.dim() == 2 else int(g.shape[0]) for g in G}
    if len(ks) > 1:
        raise ValueError("every G[i] must stack the same number of gradients")
    for w, g in zip(W, G):
        if tuple(g.shape[-2:]) != tuple(w.shape):
            raise ValueError("G[i] must match W[i]'s shape (optionally with a leading stack dimension)")
    return ks.pop() if ks else 1


def _opts(W, G, steps, coeffs, eps, nesterov, workspace, o_out=None, fp8_gram=False):
    o = _Opts()
    lib().muon_step_opts_init(ctypes.byref(o))
    o.g_count = _g_count(W, G)
    o.ns_fp8_gram = 1 if fp8_gram else 0
    o.w_dtype = _dtype_code(W[0]) if W else MUON_BF16
    o.g_dtype = _dtype_code(G[0]) if G else MUON_BF16
    o.steps = int(steps)
    o.eps = float(eps)
    o.nesterov = 1 if nesterov else 0
    carr, per_step = _schedule(coeffs, int(steps))
    if carr is not None:
        o.coeffs = ctypes.cast(carr, ctypes.POINTER(ctypes.c_float))
        o.coeffs_per_step = per_step
    if workspace is not None:
        if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        _check_device("workspace", workspace)
        o.workspace = ctypes.c_void_p(workspace.data_ptr())
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    oarr = None
    if o_out is not None:
        o_out = list(o_out)
        _check_mats("o_out", o_out, (torch.bfloat16,))
        if len(o_out) != len(W) or any(tuple(a.shape) != tuple(b.shape) for a, b in zip(o_out, W)):
            raise ValueError("o_out must match W's shapes")
        oarr = _ptr_array(o_out)
        o.o_out = ctypes.cast(oarr, ctypes.POINTER(ctypes.c_void_p))
    return o, (carr, oarr)


def muon_step_ex(W, G, M, lr: float, mu: float, wd: float, *, steps: int = 5, coeffs=None,
                 eps: float = 1e-7, nesterov: bool = True, workspace=None, o_out=None,
                 fp8_gram: bool = False, stream=None) -> None:
    """Muon step with explicit options; W and G may each be bf16 or fp32.
    ``o_out``: optional list of bf16 CUDA tensors shaped like W receiving O.
    ``fp8_gram``: the FP8 variant (E4M3 operands in the Gram product of the
    tensor-core matrices)."""
    W, G, M = list(W), list(G), list(M)
    _check_step_shapes(W, G, M, stacked_g=True)
    _check_mats("W", W, (torch.bfloat16, torch.float32))
    _check_mats("G", G, (torch.bfloat16, torch.float32), stacked=True)
    _check_mats("M", M, (torch.float32,))
    _check_one_dtype(W, G)
    rows, cols = _dims(W)
    o, _keep = _opts(W, G, steps, coeffs, eps, nesterov, workspace, o_out, fp8_gram)
    _check(lib().muon_step_ex(_ptr_array(W), _ptr_array(G), _ptr_array(M), rows, cols, len(W),
                              float(lr), float(mu), float(wd), ctypes.byref(o),
                              _stream_handle(stream)))


def _check_one_dtype(W, G):
    if W and any(t.dtype != W[0].dtype for t in W):
        raise ValueError("every W must have the same dtype")
    if G and any(t.dtype != G[0].dtype for t in G):
        raise ValueError("every G must have the same dtype")


def _check_host(name, tensors, dtypes):
    for i, t in enumerate(tensors):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise ValueError(f"{name}[{i}] must be a host tensor")
        if not t.is_contiguous() or not t.is_pinned():
            raise ValueError(f"{name}[{i}] must be contiguous pinned host memory")
        if t.dtype not in dtypes:
            raise ValueError(f"{name}[{i}] has dtype {t.dtype}; expected one of {dtypes}")


class MuonHostStep:
    """Pre-marshalled arguments for repeated Muon steps on host-resident
    (pinned) W, G, M; each ``step()`` is one muon_step_host call."""

    def __init__(self, W, G, M, *, steps: int = 5, coeffs=None, eps: float = 1e-7,
                 nesterov: bool = True):
        self.W, self.G, self.M = list(W), list(G), list(M)
        _check_step_shapes(self.W, self.G, self.M, stacked_g=True)
        _check_host("W", self.W, (torch.bfloat16, torch.float32))
        _check_host("G", self.G, (torch.bfloat16, torch.float32))
        _check_host("M", self.M, (torch.float32,))
        _check_one_dtype(self.W, self.G)
        self._w, self._g, self._m = _ptr_array(self.W), _ptr_array(self.G), _ptr_array(self.M)
        self._rows, self._cols = _dims(self.W)
        self._opts, self._keep = _opts(self.W, self.G, steps, coeffs, eps, nesterov, None)

    def step(self, lr: float, mu: float, wd: float, stream=None) -> None:
        _check(lib().muon_step_host(self._w, self._g, self._m, self._rows, self._cols, len(self.W),
                                    float(lr), float(mu), float(wd), ctypes.byref(self._opts),
                                    _stream_handle(stream)))


def muon_step_host(W, G, M, lr: float, mu: float, wd: float, *, steps: int = 5, coeffs=None,
                   eps: float = 1e-7, nesterov: bool = True, stream=None) -> None:
    """Muon step on pinned host tensors (optimizer state kept in host memory)."""
    MuonHostStep(W, G, M, steps=steps, coeffs=coeffs, eps=eps, nesterov=nesterov).step(lr, mu, wd, stream)


def muon_adamw_step(P, G, M, V, *, lr: float, beta1: float = 0.9, beta2: float = 0.95,
                    eps: float = 1e-8, wd: float = 0.0, step: int, stream=None) -> None:
    """AdamW on a list of CUDA tensors (any shape, contiguous; P and G bf16 or
    fp32, M and V fp32); ``step`` is the 1-based step number."""
    P, G, M, V = list(P), list(G), list(M), list(V)
    if not (len(P) == len(G) == len(M) == len(V)):
        raise ValueError("P, G, M and V must have the same length")
    device = None
    for name, L, dts in (("P", P, (torch.bfloat16, torch.float32)), ("G", G, (torch.bfloat16, torch.float32)),
                         ("M", M, (torch.float32,)), ("V", V, (torch.float32,))):
        for i, t in enumerate(L):
            if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous() or t.dtype not in dts:
                raise ValueError(f"{name}[{i}] must be a contiguous CUDA tensor of {dts}")
            device = _check_device(f"{name}[{i}]", t, device)
            if t.numel() != P[i].numel():
                raise ValueError(f"{name}[{i}] has {t.numel()} elements; P[{i}] has {P[i].numel()}")
    if P and any(t.dtype != P[0].dtype for t in P) or G and any(t.dtype != G[0].dtype for t in G):
        raise ValueError("every P (and every G) must share one dtype")
    n = len(P)
    numel = (ctypes.c_longlong * max(1, n))(*[t.numel() for t in P])
    pd = _dtype_code(P[0]) if P else MUON_BF16
    gd = _dtype_code(G[0]) if G else MUON_BF16
    _check(lib().muon_adamw_step(_ptr_array(P), _ptr_array(G), _ptr_array(M), _ptr_array(V), numel, n, pd, gd,
                                 float(lr), float(beta1), float(beta2), float(eps), float(wd), int(step),
                                 _stream_handle(stream)))


def muon_workspace_bytes(shapes) -> int:
    shapes = list(shapes)
    n = len(shapes)
    rows = (ctypes.c_int * max(n, 1))(*[int(s[0]) for s in shapes])
    cols = (ctypes.c_int * max(n, 1))(*[int(s[1]) for s in shapes])
    return int(lib().muon_workspace_bytes(rows, cols, n))


def muon_device_status(stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().muon_device_status(_stream_handle(stream), ctypes.byref(st)))
    return st.value


def muon_release_workspace() -> None:
    lib().muon_release_workspace()


def muon_profile_enable(on: bool = True) -> None:
    _check(lib().muon_profile_enable(1 if on else 0))


def muon_profile_read():
    arr = (_KernelStat * 16)()
    n = ctypes.c_int(0)
    _check(lib().muon_profile_read(arr, 16, ctypes.byref(n)))
    return [{"name": arr[i].name.decode(), "launches": arr[i].launches, "total_ms": arr[i].total_ms,
             "flops": arr[i].flops, "bytes": arr[i].bytes} for i in range(n.value)]


class MuonStepBatch:
    """Pre-marshalled arguments for repeated Muon steps on the same tensors.

    Builds the pointer and dimension arrays once; ``step()`` then makes one
    C call per optimizer step.
    """

    def __init__(self, W, G, M, *, steps: int = 5, coeffs=None, eps: float = 1e-7,
                 nesterov: bool = True, workspace=None, fp8_gram: bool = False):
        self.W, self.G, self.M = list(W), list(G), list(M)
        _check_step_shapes(self.W, self.G, self.M, stacked_g=True)
        _check_mats("W", self.W, (torch.bfloat16, torch.float32))
        _check_mats("G", self.G, (torch.bfloat16, torch.float32), stacked=True)
        _check_mats("M", self.M, (torch.float32,))
        _check_one_dtype(self.W, self.G)
        self._w, self._g, self._m = _ptr_array(self.W), _ptr_array(self.G), _ptr_array(self.M)
        self._rows, self._cols = _dims(self.W)
        self._opts, self._keep = _opts(self.W, self.G, steps, coeffs, eps, nesterov, workspace, None, fp8_gram)

    def step(self, lr: float, mu: float, wd: float, stream=None) -> None:
        _check(lib().muon_step_ex(self._w, self._g, self._m, self._rows, self._cols, len(self.W),
                                  float(lr), float(mu), float(wd), ctypes.byref(self._opts),
                                  _stream_handle(stream)))
