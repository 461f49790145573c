"""CPU oracle for the per-matrix Muon step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The CUDA library never calls it and
shares no code with it; the two meet only through the seeded input generators
(``muon_newton_schulz_step_gb300.workloads``), which hold none of the method's
arithmetic.

The arithmetic lives in ``muon_oracle.c`` (plain C, see its header for the
formulas and the readings taken where "How PyTorch Scaled a Near-1T MoE on
Europe's Public Supercomputer" -- section "Three optimizations that changed the
economics", FlexShard bullet -- leaves a step open).  This module only marshals
numpy arrays to it.  bf16 tensors travel as ``uint16`` bit patterns.

Parity status of each function (what pins it in ``tests/test_oracle_*.py``):
  bf16_rne          pinned: torch's round-to-nearest-even cast, edge values
  momentum          pinned: exact rational arithmetic (fractions.Fraction)
  ns (f64 mode)     pinned: closed form U p^5(s/|s|) V^T from an SVD; special
                    cases (rank 1, c*I, zero); brute-force shapes
  ns (bf16 mode)    pinned: closed form within the bf16 error scale, the
                    singular-value band invariant, exactness on matrices
                    whose every intermediate is bf16-representable
  update            pinned: exact rational arithmetic
  grad_sum          pinned: exact rational arithmetic
  ns_schedule       pinned: closed form with the composed per-step polynomials
  adamw             pinned: torch.optim.AdamW in fp64 (an independent library
                    implementation), the first-step closed form, zero gradient
  e4m3_rne          pinned: torch's float8_e4m3fn cast (an independent library
                    implementation) on every in-range magnitude grid, ties,
                    subnormals; saturation and NaN by the format's definition
  ns_fp8_gram       pinned: equals the bf16 mode bit for bit where every X is
                    E4M3-representable after scaling; closed form within the
                    FP8 error scale; distance from the bf16 mode bounded
"""
import ctypes
import os

import numpy as np

from . import build as _build

COEFFS = (3.4445, -4.7750, 2.0315)
EPS = 1e-7

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        L.oracle_bf16_rne.restype = ctypes.c_uint16
        L.oracle_bf16_rne.argtypes = [ctypes.c_float]
        L.oracle_bf16_rne_array.restype = None
        L.oracle_bf16_rne_array.argtypes = [f32p, u16p, ctypes.c_int64]
        L.oracle_grad_sum.restype = None
        L.oracle_grad_sum.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, f32p]
        L.oracle_momentum.restype = None
        L.oracle_momentum.argtypes = [f32p, f32p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_int]
        L.oracle_ns_bf16.restype = ctypes.c_int
        L.oracle_ns_bf16.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                     ctypes.c_double, f32p]
        L.oracle_ns_bf16_sched.restype = ctypes.c_int
        L.oracle_ns_bf16_sched.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32p,
                                           ctypes.c_double, f32p]
        L.oracle_ns_f64_sched.restype = ctypes.c_int
        L.oracle_ns_f64_sched.argtypes = [f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, f64p,
                                          ctypes.c_double, f64p]
        L.oracle_ns_f64.restype = ctypes.c_int
        L.oracle_ns_f64.argtypes = [f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, f64p]
        L.oracle_update_scalars.restype = None
        L.oracle_update_scalars.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                            ctypes.c_int, f32p, f32p]
        L.oracle_weight_update_f32.restype = None
        L.oracle_weight_update_f32.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_float]
        L.oracle_weight_update_bf16.restype = None
        L.oracle_weight_update_bf16.argtypes = [u16p, f32p, ctypes.c_int64, ctypes.c_float, ctypes.c_float]
        L.oracle_adamw.restype = None
        L.oracle_adamw.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, f32p, f32p,
                                   ctypes.c_int64, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                   ctypes.c_float, ctypes.c_float, ctypes.c_int]
        L.oracle_adamw_scalars.restype = None
        L.oracle_adamw_scalars.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int, f32p]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_e4m3_rne.restype = ctypes.c_uint8
        L.oracle_e4m3_rne.argtypes = [ctypes.c_float]
        L.oracle_e4m3_to_f32.restype = ctypes.c_float
        L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_rne_array.restype = None
        L.oracle_e4m3_rne_array.argtypes = [f32p, u8p, ctypes.c_int64]
        L.oracle_ns_bf16_sched_fp8.restype = ctypes.c_int
        L.oracle_ns_bf16_sched_fp8.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32p,
                                               ctypes.c_double, f32p]
        L.oracle_set_sum_order.restype = None
        L.oracle_set_sum_order.argtypes = [ctypes.c_int]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_num_threads.argtypes = []
        _lib = L
    return _lib


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(lib().oracle_num_threads())


class descending_sums:
    """Context manager: inside it, the bf16-emulating products sum over p in
    descending instead of ascending order.  Both orders are valid readings
    (the pages fix none); the switch exists only to measure how far a legal
    change of summation order moves a result, i.e. how ill-conditioned an input
    is.  Parity checks always use the default ascending order."""

    def __enter__(self):
        lib().oracle_set_sum_order(1)
        return self

    def __exit__(self, *exc):
        lib().oracle_set_sum_order(0)
        return False


# ---------------------------------------------------------------- bf16 ----
def bf16_rne(x) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_bf16_rne_array(_p(x, ctypes.c_float), _p(out, ctypes.c_uint16), x.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- e4m3 ----
def e4m3_rne(x) -> np.ndarray:
    """fp32 array -> FP8 E4M3 codes (uint8), round to nearest even, saturating."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_rne_array(_p(x, ctypes.c_float), _p(out, ctypes.c_uint8), x.size)
    return out


def e4m3_to_f32(codes) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    return np.array([lib().oracle_e4m3_to_f32(int(v)) for v in codes.ravel()], dtype=np.float32).reshape(codes.shape)


# ------------------------------------------------- gradient accumulation ----
def grad_sum(G_stack, g_bf16: bool) -> np.ndarray:
    """fp32 sum, in order, of K stacked gradients (K x m x n; bf16 bits or fp32)."""
    G = np.ascontiguousarray(G_stack, dtype=np.uint16 if g_bf16 else np.float32)
    K = G.shape[0]
    out = np.empty(G.shape[1:], dtype=np.float32)
    lib().oracle_grad_sum(G.ctypes.data_as(ctypes.c_void_p), int(bool(g_bf16)), out.size, K,
                          _p(out, ctypes.c_float))
    return out


# ------------------------------------------------------------ momentum ----
def momentum(g, M, mu: float, nesterov: bool = True):
    """Returns (M', U) for fp32 g and M (M is not modified)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    Mn = np.array(M, dtype=np.float32, copy=True, order="C")
    U = np.empty_like(Mn)
    lib().oracle_momentum(_p(g, ctypes.c_float), _p(Mn, ctypes.c_float), _p(U, ctypes.c_float),
                          g.size, np.float32(mu), int(bool(nesterov)))
    return Mn, U


# ------------------------------------------------------- Newton-Schulz ----
def ns(U, steps: int = 5, coeffs=COEFFS, eps: float = EPS, mode: str = "bf16") -> np.ndarray:
    """Normalise + Newton-Schulz one 2-D matrix.

    mode "bf16": fp32 input, bf16-emulated iterate, returns fp32 (bf16-exact).
    mode "f64":  fp64 throughout, no rounding, returns fp64.
    """
    a, b, c = coeffs
    if mode == "bf16":
        U = np.ascontiguousarray(U, dtype=np.float32)
        m, n = U.shape
        O = np.empty_like(U)
        rc = lib().oracle_ns_bf16(_p(U, ctypes.c_float), m, n, int(steps),
                                  np.float32(a), np.float32(b), np.float32(c), float(eps),
                                  _p(O, ctypes.c_float))
    elif mode == "f64":
        U = np.ascontiguousarray(U, dtype=np.float64)
        m, n = U.shape
        O = np.empty_like(U)
        rc = lib().oracle_ns_f64(_p(U, ctypes.c_double), m, n, int(steps),
                                 float(a), float(b), float(c), float(eps),
                                 _p(O, ctypes.c_double))
    else:
        raise ValueError(mode)
    if rc != 0:
        raise RuntimeError("oracle_ns failed")
    return O


def ns_schedule(U, schedule, eps: float = EPS, mode: str = "bf16") -> np.ndarray:
    """Normalise + Newton-Schulz with one (a, b, c) triple per step
    (``schedule`` is a sequence of triples; its length is the step count)."""
    sched = np.asarray(schedule, dtype=np.float64).reshape(-1, 3)
    steps = sched.shape[0]
    if mode == "bf16":
        U = np.ascontiguousarray(U, dtype=np.float32)
        m, n = U.shape
        O = np.empty_like(U)
        abc = np.ascontiguousarray(sched.astype(np.float32).ravel())
        if abc.size == 0:
            abc = np.zeros(3, dtype=np.float32)
        rc = lib().oracle_ns_bf16_sched(_p(U, ctypes.c_float), m, n, steps, _p(abc, ctypes.c_float),
                                        float(eps), _p(O, ctypes.c_float))
    elif mode == "f64":
        U = np.ascontiguousarray(U, dtype=np.float64)
        m, n = U.shape
        O = np.empty_like(U)
        abc = np.ascontiguousarray(sched.ravel()) if sched.size else np.zeros(3)
        rc = lib().oracle_ns_f64_sched(_p(U, ctypes.c_double), m, n, steps, _p(abc, ctypes.c_double),
                                       float(eps), _p(O, ctypes.c_double))
    else:
        raise ValueError(mode)
    if rc != 0:
        raise RuntimeError("oracle_ns_schedule failed")
    return O


def ns_fp8_gram(U, steps: int = 5, coeffs=COEFFS, eps: float = EPS, schedule=None) -> np.ndarray:
    """Normalise + Newton-Schulz in the FP8 variant: the Gram product's
    operands are X * 2^8 rounded to E4M3 (an exact scaling; the iterates stay
    below 1.21, so nothing saturates), the sum unscaled by 2^-16 (fp32 input,
    bf16-emulated iterate, returns fp32)."""
    sched = np.asarray(schedule if schedule is not None else [coeffs] * steps, dtype=np.float64).reshape(-1, 3)
    U = np.ascontiguousarray(U, dtype=np.float32)
    m, n = U.shape
    O = np.empty_like(U)
    abc = np.ascontiguousarray(sched.astype(np.float32).ravel()) if sched.size else np.zeros(3, dtype=np.float32)
    rc = lib().oracle_ns_bf16_sched_fp8(_p(U, ctypes.c_float), m, n, sched.shape[0], _p(abc, ctypes.c_float),
                                        float(eps), _p(O, ctypes.c_float))
    if rc != 0:
        raise RuntimeError("oracle_ns_fp8_gram failed")
    return O


def ns_bf16_bits(X_bits, steps: int = 5, coeffs=COEFFS, eps: float = EPS) -> np.ndarray:
    """In-place-style NS of a bf16 matrix given as uint16 bits; returns bf16 bits."""
    O = ns(bf16_to_f32(X_bits), steps, coeffs, eps, mode="bf16")
    return bf16_rne(O)


# -------------------------------------------------------------- update ----
def update_scalars(lr: float, wd: float, m: int, n: int):
    dcy = ctypes.c_float()
    s = ctypes.c_float()
    lib().oracle_update_scalars(np.float32(lr), np.float32(wd), int(m), int(n),
                                ctypes.byref(dcy), ctypes.byref(s))
    return np.float32(dcy.value), np.float32(s.value)


def weight_update(W, O, dcy, s, w_bf16: bool):
    """Returns the updated W (bf16 bits if w_bf16 else fp32); W is not modified."""
    O = np.ascontiguousarray(O, dtype=np.float32)
    if w_bf16:
        Wn = np.array(W, dtype=np.uint16, copy=True, order="C")
        lib().oracle_weight_update_bf16(_p(Wn, ctypes.c_uint16), _p(O, ctypes.c_float), O.size,
                                        np.float32(dcy), np.float32(s))
    else:
        Wn = np.array(W, dtype=np.float32, copy=True, order="C")
        lib().oracle_weight_update_f32(_p(Wn, ctypes.c_float), _p(O, ctypes.c_float), O.size,
                                       np.float32(dcy), np.float32(s))
    return Wn


# ----------------------------------------------------------- full step ----
def muon_step(W, G, M, lr, mu, wd, *, w_bf16: bool, g_bf16: bool, nesterov: bool = True,
              steps: int = 5, coeffs=COEFFS, eps: float = EPS, schedule=None, fp8_gram: bool = False):
    """One Muon step on one matrix.  Returns (W', M', O) without modifying inputs.

    W: bf16 bits (w_bf16) or fp32;  G: bf16 bits (g_bf16) or fp32, either one
    m x n gradient or a K x m x n stack that is summed in fp32 first;  M: fp32.
    O is the orthogonalised update as fp32 (bf16-exact values).  ``schedule``
    (one (a, b, c) per step) replaces steps/coeffs when given.
    """
    if np.ndim(G) == 3:
        g = grad_sum(G, g_bf16)
    else:
        g = bf16_to_f32(G) if g_bf16 else np.ascontiguousarray(G, dtype=np.float32)
    M1, U = momentum(g, M, mu, nesterov)
    if fp8_gram:
        O = ns_fp8_gram(U, steps, coeffs, eps, schedule)
    else:
        O = ns_schedule(U, schedule, eps) if schedule is not None else ns(U, steps, coeffs, eps, mode="bf16")
    m, n = O.shape
    dcy, s = update_scalars(lr, wd, m, n)
    W1 = weight_update(W, O, dcy, s, w_bf16)
    return W1, M1, O


# ---------------------------------------------------------------- AdamW ----
def adamw(P, G, M, V, *, lr, beta1, beta2, eps, wd, step, p_bf16: bool, g_bf16: bool):
    """One AdamW step on a flat parameter.  Returns (P', M', V') without
    modifying the inputs.  P, G: bf16 bits or fp32;  M, V: fp32."""
    Pn = np.array(P, dtype=np.uint16 if p_bf16 else np.float32, copy=True, order="C").ravel()
    Gc = np.ascontiguousarray(G, dtype=np.uint16 if g_bf16 else np.float32).ravel()
    Mn = np.array(M, dtype=np.float32, copy=True, order="C").ravel()
    Vn = np.array(V, dtype=np.float32, copy=True, order="C").ravel()
    lib().oracle_adamw(Pn.ctypes.data_as(ctypes.c_void_p), int(p_bf16), Gc.ctypes.data_as(ctypes.c_void_p),
                       int(g_bf16), _p(Mn, ctypes.c_float), _p(Vn, ctypes.c_float), Pn.size,
                       np.float32(lr), np.float32(beta1), np.float32(beta2), np.float32(eps),
                       np.float32(wd), int(step))
    return Pn, Mn, Vn


def adamw_scalars(lr, beta1, beta2, wd, step):
    out = np.empty(5, dtype=np.float32)
    lib().oracle_adamw_scalars(np.float32(lr), np.float32(beta1), np.float32(beta2), np.float32(wd),
                               int(step), _p(out, ctypes.c_float))
    return out
