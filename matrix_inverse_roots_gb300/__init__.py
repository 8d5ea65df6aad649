"""Python binding of dashroot, the GB300 library for the batched block-preconditioner
step of DASH-style Shampoo (factor accumulation, spectral scaling, inverse 4th
roots by Coupled Newton / Newton-Denman-Beavers / Chebyshev-Clenshaw, and the
preconditioned update).

This module only marshals arguments: it checks tensor shapes and dtypes, passes
raw device pointers and the current CUDA stream to the C ABI declared in
``include/dashroot.h``, and allocates workspaces with PyTorch.  Every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if
``libdashroot.so`` is missing the first call raises.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdashroot.so")

# dash_prec
FP32_3XTF32 = 0
TF32 = 1
FP16 = 2
BF16 = 3
PRECISIONS = {"3xtf32": FP32_3XTF32, "fp32": FP32_3XTF32, "tf32": TF32, "fp16": FP16,
              "bf16": BF16}
# Flag OR-ed into prec (DASH_ROOT_TF32): root solvers write X rounded to TF32;
# precondition_apply / _update with TF32 then read such roots without converting.
ROOT_TF32 = 0x100

# dash_dtype
DT_F32 = 0
DT_BF16 = 1
DT_F16 = 2

# dash_scale_mode
SCALE_POWER = 0
SCALE_FROBENIUS = 1
SCALE_POWER_F16 = 2
SCALE_POWER_BF16 = 3
_HALF_SCALE = {SCALE_POWER_F16: FP16, SCALE_POWER_BF16: BF16}

# dash_solver
SOLVER_CN = 0
SOLVER_NDB = 1
SOLVER_CHEB = 2
SOLVERS = {"cn": SOLVER_CN, "ndb": SOLVER_NDB, "cheb": SOLVER_CHEB}


class Tier(ctypes.Structure):
    """dash_tier: one tier of per-block solver selection."""
    _fields_ = [("solver", ctypes.c_int), ("prec", ctypes.c_int), ("iters", ctypes.c_int),
                ("u", ctypes.c_double), ("gate", ctypes.c_double)]


# Default tiers of per-block solver selection, cheapest first: Coupled Newton in
# FP16 (10 iterations, unit roundoff of fp16 storage, the 1e-2 FP16 tolerance),
# else Coupled Newton in 3xTF32 with 24 iterations, enough for a smallest scaled
# eigenvalue of 1e-6 to converge (each early iteration multiplies it by about
# (5/4)^4), held to the 1e-4 fp32 tolerance.
DEFAULT_TIERS = (
    {"solver": "cn", "prec": "fp16", "iters": 10, "u": 2.0 ** -11, "gate": 1e-2},
    {"solver": "cn", "prec": "3xtf32", "iters": 24, "u": 2.0 ** -24, "gate": 1e-4},
)


# dash_op
OP_ACCUMULATE = 0
OP_SPECTRAL_SCALE = 1
OP_INV_ROOT_CN = 2
OP_INV_ROOT_NDB = 3
OP_INV_ROOT_CHEB = 4
OP_PRECONDITION_APPLY = 5
OP_LAMBDA_MIN = 6

# Exported C symbols (kept in step with include/dashroot.h).
SYMBOLS = (
    "shampoo_accumulate", "spectral_scale", "inv_root_cn", "inv_root_ndb", "inv_root_cheb",
    "precondition_apply", "dash_gemm", "dash_workspace_size", "dash_op_matmuls",
    "dash_device_status", "dash_status_string", "dash_version", "dash_trace_start",
    "dash_trace_count", "dash_trace_read", "dash_trace_stop", "spectral_scale_noalloc",
    "dash_selftest_wait_timeout", "precondition_update", "pack_blocks", "unpack_blocks",
    "dash_cheb_coeffs", "dash_select_tiers", "spectral_lambda_min", "inv_root_auto",
    "dash_auto_workspace_size", "dash_gemm_ex",
)

_lib = None


class DashError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s" % (what, status_string(status)))


def load_library(path=None):
    """Load libdashroot.so (raises OSError if it was not built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError("libdashroot.so not found at %s: build it with "
                      "`python -m matrix_inverse_roots_gb300.build`" % p)
    lib = ctypes.CDLL(p)
    vp, i64, i32, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
    lib.shampoo_accumulate.argtypes = [vp, i32, i64, i32, f32, vp, vp, vp, vp, sz, vp]
    lib.spectral_scale.argtypes = [vp, f32, i64, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.inv_root_cn.argtypes = [vp, f32, vp, i64, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.inv_root_ndb.argtypes = [vp, f32, vp, i64, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.inv_root_cheb.argtypes = [vp, f32, vp, i64, i32, i32, f64, f64, i32, vp, vp, sz, vp]
    lib.precondition_apply.argtypes = [vp, i32, vp, i64, i32, i32, vp, vp, sz, vp]
    lib.precondition_update.argtypes = [vp, i32, vp, i64, i32, i32, f32, vp, vp, vp, sz, vp]
    lib.pack_blocks.argtypes = [vp, i32, i64, i64, i64, i32, vp, vp, vp, vp]
    lib.unpack_blocks.argtypes = [vp, i32, i64, i64, i64, i32, vp, vp]
    lib.dash_gemm.argtypes = [vp, vp, i32, vp, vp, i32, i64, i32, i32, vp, vp]
    lib.dash_workspace_size.argtypes = [i32, i64, i32, i32, i32, ctypes.POINTER(sz)]
    lib.dash_op_matmuls.argtypes = [i32, i32]
    lib.dash_op_matmuls.restype = i64
    lib.dash_device_status.argtypes = []
    lib.dash_status_string.argtypes = [i32]
    lib.dash_status_string.restype = ctypes.c_char_p
    lib.dash_version.restype = ctypes.c_char_p
    lib.spectral_scale_noalloc.argtypes = [vp, f32, i64, i32, i32, i32, i32, vp, vp, vp]
    lib.spectral_scale_noalloc.restype = ctypes.c_int
    lib.dash_cheb_coeffs.argtypes = [i32, f64, f64, ctypes.POINTER(f64)]
    lib.dash_select_tiers.argtypes = [ctypes.POINTER(f32), ctypes.POINTER(f32), i64,
                                      ctypes.POINTER(Tier), i32, ctypes.POINTER(ctypes.c_int32)]
    lib.dash_select_tiers.restype = ctypes.c_int
    lib.spectral_lambda_min.argtypes = [vp, f32, vp, i64, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.spectral_lambda_min.restype = ctypes.c_int
    lib.inv_root_auto.argtypes = [vp, f32, vp, vp, i64, i32, ctypes.POINTER(Tier), i32, f64, f64,
                                  vp, ctypes.POINTER(ctypes.c_int32), vp, sz, vp]
    lib.inv_root_auto.restype = ctypes.c_int
    lib.dash_auto_workspace_size.argtypes = [i64, i32, ctypes.POINTER(Tier), i32,
                                             ctypes.POINTER(sz)]
    lib.dash_auto_workspace_size.restype = ctypes.c_int
    lib.dash_gemm_ex.argtypes = [vp, vp, i32, vp, vp, i32, i64, i32, i32, i32, vp, vp]
    lib.dash_gemm_ex.restype = ctypes.c_int
    lib.dash_cheb_coeffs.restype = ctypes.c_int
    lib.dash_selftest_wait_timeout.argtypes = [i32, vp]
    lib.dash_selftest_wait_timeout.restype = ctypes.c_int
    lib.dash_trace_start.argtypes = [i32]
    lib.dash_trace_count.argtypes = []
    lib.dash_trace_count.restype = i32
    lib.dash_trace_read.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(f64),
                                    ctypes.POINTER(f64), ctypes.POINTER(f32)]
    lib.dash_trace_stop.argtypes = []
    for name in ("shampoo_accumulate", "spectral_scale", "inv_root_cn", "inv_root_ndb",
                 "inv_root_cheb", "precondition_apply", "precondition_update", "pack_blocks",
                 "unpack_blocks", "dash_gemm", "dash_workspace_size",
                 "dash_device_status", "dash_trace_start", "dash_trace_read", "dash_trace_stop"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(status):
    try:
        return load_library().dash_status_string(int(status)).decode()
    except OSError:
        return "status %d" % status


def _check(status, what):
    if status != 0:
        raise DashError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _stack(t, name, dtype=torch.float32):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    # The library launches on the current device's stream (and the no-allocation
    # entry point uses that device's built-in scratch): a tensor elsewhere would be
    # handed to kernels of the wrong device.
    if t.device.index != torch.cuda.current_device():
        raise ValueError("%s is on %s but the current CUDA device is cuda:%d" % (
            name, t.device, torch.cuda.current_device()))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _shape(t, shape, name):
    """Sizes the kernels will index: a wrong one would read or write past t."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _blocks3(t, name):
    if t.dim() != 3 or t.shape[1] != t.shape[2]:
        raise ValueError("%s must be a (N, B, B) stack, got %s" % (name, tuple(t.shape)))
    return t.shape[0], t.shape[1]


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def _gdt(t):
    if t.dtype == torch.float32:
        return DT_F32
    if t.dtype == torch.bfloat16:
        return DT_BF16
    if t.dtype == torch.float16:
        return DT_F16
    raise TypeError("gradient dtype must be float32, bfloat16 or float16")


def _prec(p):
    """A precision name ("fp16", ...; "+root_tf32" adds ROOT_TF32) or a dash_prec value."""
    if isinstance(p, str):
        name, _, flag = p.lower().partition("+")
        if flag not in ("", "root_tf32"):
            raise ValueError("unknown precision flag %r" % flag)
        return PRECISIONS[name] | (ROOT_TF32 if flag else 0)
    return int(p)


def version():
    return load_library().dash_version().decode()


def workspace_size(op, n, b, prec=FP32_3XTF32, param=0):
    out = ctypes.c_size_t(0)
    _check(load_library().dash_workspace_size(int(op), int(n), int(b), _prec(prec), int(param),
                                              ctypes.byref(out)), "dash_workspace_size")
    return out.value


def workspace(op, n, b, prec=FP32_3XTF32, param=0, device=None, max_bytes=None):
    """Allocate a workspace with PyTorch (optionally capped at max_bytes)."""
    nbytes = workspace_size(op, n, b, prec, param)
    if max_bytes is not None:
        nbytes = min(nbytes, int(max_bytes))
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


# dash_trace_kind
TRACE_KINDS = ("gemm_f16", "gemm_bf16", "gemm_tf32", "gemm_3xtf32", "elementwise", "power",
               "reduce", "pack")


def trace_start(capacity=4096):
    """Record CUDA events around every library kernel launch from now on."""
    _check(load_library().dash_trace_start(int(capacity)), "dash_trace_start")


def trace_stop():
    _check(load_library().dash_trace_stop(), "dash_trace_stop")


def trace_records():
    """[(kind name, algorithmic flops, algorithmic bytes, device ms)] of the trace."""
    lib = load_library()
    out = []
    k = ctypes.c_int(0)
    fl = ctypes.c_double(0)
    by = ctypes.c_double(0)
    ms = ctypes.c_float(0)
    for i in range(lib.dash_trace_count()):
        _check(lib.dash_trace_read(i, ctypes.byref(k), ctypes.byref(fl), ctypes.byref(by),
                                   ctypes.byref(ms)), "dash_trace_read")
        out.append((TRACE_KINDS[k.value], fl.value, by.value, ms.value))
    return out


def cheb_coeffs(degree, lo=1e-2, hi=1.05):
    """The Chebyshev coefficients inv_root_cheb uses (computed on the host)."""
    c = (ctypes.c_double * (int(degree) + 1))()
    _check(load_library().dash_cheb_coeffs(int(degree), float(lo), float(hi), c),
           "dash_cheb_coeffs")
    return list(c)


def select_tiers(lam_max, lam_min, tiers):
    """Tier index per block from host sequences of lambda_max / lambda_min estimates.

    tiers: sequence of dicts with keys solver ("cn" | "ndb" | "cheb"), prec, iters,
    u, gate (cheapest first).  Host-side: no GPU is used."""
    lmax = [float(x) for x in lam_max]
    lmin = [float(x) for x in lam_min]
    if len(lmax) != len(lmin):
        raise ValueError("lam_max and lam_min must have the same length")
    n = len(lmax)
    tt = _tiers(tiers)
    a = (ctypes.c_float * max(n, 1))(*lmax)
    b = (ctypes.c_float * max(n, 1))(*lmin)
    out = (ctypes.c_int32 * max(n, 1))()
    _check(load_library().dash_select_tiers(a, b, n, tt, len(tiers), out), "dash_select_tiers")
    return list(out)[:n]


def _tiers(tiers):
    return (Tier * len(tiers))(*[Tier(SOLVERS[t["solver"]], _prec(t["prec"]), int(t["iters"]),
                                      float(t["u"]), float(t["gate"])) for t in tiers])


def spectral_lambda_min(A, lam_max, mode=SCALE_POWER, V0=None, power_iters=10, ridge=0.0,
                        out=None, ws=None):
    """lambda_min estimate per block: power iteration on lam_max I - (A + ridge I)."""
    lib = load_library()
    _stack(A, "A")
    n, b = _blocks3(A, "A")
    _shape(_stack(lam_max, "lam_max"), (n,), "lam_max")
    _stack(V0, "V0")
    if V0.dim() != 3 or V0.shape[0] != n or V0.shape[1] != b:
        raise ValueError("V0 must have shape (N, B, n_vec)")
    nv = V0.shape[2]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=A.device)
    _shape(_stack(out, "out"), (n,), "out")
    if ws is None:
        ws = workspace(OP_LAMBDA_MIN, n, b, _HALF_SCALE.get(mode, FP32_3XTF32), nv,
                       device=A.device)
    _check(lib.spectral_lambda_min(_ptr(A), float(ridge), _ptr(lam_max), n, b, int(mode), nv,
                                   int(power_iters), _ptr(V0), _ptr(out), _ptr(ws), _nbytes(ws),
                                   _stream()), "spectral_lambda_min")
    return out


def auto_workspace_size(n, b, tiers):
    out = ctypes.c_size_t(0)
    tt = _tiers(tiers)
    _check(load_library().dash_auto_workspace_size(int(n), int(b), tt, len(tiers),
                                                   ctypes.byref(out)), "dash_auto_workspace_size")
    return out.value


def inv_root_auto(A, lam_max, lam_min, tiers, ridge=0.0, cheb=(1e-2, 1.05), X=None, ws=None,
                  max_ws_bytes=None):
    """A^{-1/4} with the solver chosen per block by its condition estimate.

    tiers: sequence of dicts (solver, prec, iters, u, gate), cheapest first.  Returns
    (X, choice) with choice the list of tier indices.  Synchronises the stream (the
    estimates are read back to the host)."""
    lib = load_library()
    _stack(A, "A")
    n, b = _blocks3(A, "A")
    _shape(_stack(lam_max, "lam_max"), (n,), "lam_max")
    _shape(_stack(lam_min, "lam_min"), (n,), "lam_min")
    if X is None:
        X = torch.empty_like(A)
    _shape(_stack(X, "X"), (n, b, b), "X")
    tt = _tiers(tiers)
    if ws is None:
        nbytes = auto_workspace_size(n, b, tiers)
        if max_ws_bytes is not None:
            nbytes = min(nbytes, int(max_ws_bytes))
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=A.device)
    choice = (ctypes.c_int32 * max(n, 1))()
    _check(lib.inv_root_auto(_ptr(A), float(ridge), _ptr(lam_max), _ptr(lam_min), n, b, tt,
                             len(tiers), float(cheb[0]), float(cheb[1]), _ptr(X), choice,
                             _ptr(ws), _nbytes(ws), _stream()), "inv_root_auto")
    return X, list(choice)[:n]


def op_matmuls(op, param):
    return int(load_library().dash_op_matmuls(int(op), int(param)))


def device_status():
    return int(load_library().dash_device_status())


def selftest_wait_timeout(limit_us=50000):
    """Run the bounded-wait self-test kernel (its wait times out on purpose)."""
    _check(load_library().dash_selftest_wait_timeout(int(limit_us), _stream()),
           "dash_selftest_wait_timeout")


def shampoo_accumulate(G, F, beta, valid_rows=None, valid_cols=None, ws=None):
    """In place: F[j] <- beta F[j] + (1-beta) G_j G_j^T, F[Ng+j] likewise with G_j^T G_j."""
    lib = load_library()
    _stack(G, "G", G.dtype)
    ng, b = _blocks3(G, "G")
    _shape(_stack(F, "F"), (2 * ng, b, b), "F")
    gdt = _gdt(G)
    if ws is None and gdt == DT_F32:
        ws = workspace(OP_ACCUMULATE, ng, b, FP32_3XTF32, device=G.device)
    vr = None if valid_rows is None else _shape(_stack(valid_rows, "valid_rows", torch.int32),
                                                (ng,), "valid_rows")
    vc = None if valid_cols is None else _shape(_stack(valid_cols, "valid_cols", torch.int32),
                                                (ng,), "valid_cols")
    _check(lib.shampoo_accumulate(_ptr(G), gdt, ng, b, float(beta), _ptr(F), _ptr(vr), _ptr(vc),
                                  _ptr(ws), _nbytes(ws), _stream()),
           "shampoo_accumulate")
    return F


def spectral_scale(A, mode=SCALE_POWER, V0=None, power_iters=10, ridge=0.0, out=None, ws=None):
    """Per-block scale: multi-vector power-iteration lambda_max or Frobenius norm."""
    lib = load_library()
    _stack(A, "A")
    n, b = _blocks3(A, "A")
    nv = 0
    if mode != SCALE_FROBENIUS:
        _stack(V0, "V0")
        if V0.dim() != 3 or V0.shape[0] != n or V0.shape[1] != b:
            raise ValueError("V0 must have shape (N, B, n_vec)")
        nv = V0.shape[2]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=A.device)
    _shape(_stack(out, "out"), (n,), "out")
    if ws is None:
        ws = workspace(OP_SPECTRAL_SCALE, n, b, _HALF_SCALE.get(mode, FP32_3XTF32), nv,
                       device=A.device)
    _check(lib.spectral_scale(_ptr(A), float(ridge), n, b, int(mode), nv, int(power_iters),
                              _ptr(V0), _ptr(out), _ptr(ws), _nbytes(ws), _stream()),
           "spectral_scale")
    return out


# Bytes of the library's built-in scratch used by spectral_scale_noalloc.
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def spectral_scale_noalloc(A, mode=SCALE_POWER, V0=None, power_iters=10, ridge=0.0, out=None):
    """spectral_scale without a workspace: for callers that may not allocate device
    memory when they run.  Scratch comes from a fixed 32 MiB array inside the
    library, so one call handles at most that much (127 blocks of 1024^2 with
    32 vectors); calls overlapping on the GPU share that array and must not run
    concurrently.  `out` lets the caller avoid this wrapper's own allocation."""
    lib = load_library()
    _stack(A, "A")
    n, b = _blocks3(A, "A")
    nv = 0
    if mode != SCALE_FROBENIUS:
        _stack(V0, "V0")
        if V0.dim() != 3 or V0.shape[0] != n or V0.shape[1] != b:
            raise ValueError("V0 must have shape (N, B, n_vec)")
        nv = V0.shape[2]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=A.device)
    _shape(_stack(out, "out"), (n,), "out")
    _check(lib.spectral_scale_noalloc(_ptr(A), float(ridge), n, b, int(mode), nv,
                                      int(power_iters), _ptr(V0), _ptr(out), _stream()),
           "spectral_scale_noalloc")
    return out


def _root_common(A, scale, X):
    _stack(A, "A")
    n, b = _blocks3(A, "A")
    _shape(_stack(scale, "scale"), (n,), "scale")
    if X is None:
        X = torch.empty_like(A)
    _shape(_stack(X, "X"), (n, b, b), "X")
    return n, b, X


def inv_root_cn(A, scale, iters=10, prec=FP32_3XTF32, ridge=0.0, X=None, resid=False, ws=None):
    """Coupled Newton A^{-1/4}; returns X or (X, resid (N, iters))."""
    lib = load_library()
    n, b, X = _root_common(A, scale, X)
    p = _prec(prec)
    r = torch.empty((n, int(iters)), dtype=torch.float32, device=A.device) if resid else None
    if ws is None:
        ws = workspace(OP_INV_ROOT_CN, n, b, p, iters, device=A.device)
    _check(lib.inv_root_cn(_ptr(A), float(ridge), _ptr(scale), n, b, int(iters), p, _ptr(X),
                           _ptr(r), _ptr(ws), _nbytes(ws), _stream()), "inv_root_cn")
    return (X, r) if resid else X


def inv_root_ndb(A, scale, iters=10, prec=FP32_3XTF32, ridge=0.0, X=None, resid=False, ws=None):
    """Newton-Denman-Beavers A^{-1/4}; returns X or (X, resid (N, 2, iters))."""
    lib = load_library()
    n, b, X = _root_common(A, scale, X)
    p = _prec(prec)
    r = torch.empty((n, 2, int(iters)), dtype=torch.float32, device=A.device) if resid else None
    if ws is None:
        ws = workspace(OP_INV_ROOT_NDB, n, b, p, iters, device=A.device)
    _check(lib.inv_root_ndb(_ptr(A), float(ridge), _ptr(scale), n, b, int(iters), p, _ptr(X),
                            _ptr(r), _ptr(ws), _nbytes(ws), _stream()), "inv_root_ndb")
    return (X, r) if resid else X


def inv_root_cheb(A, scale, degree=16, lo=1e-2, hi=1.05, prec=FP32_3XTF32, ridge=0.0, X=None,
                  ws=None):
    """Chebyshev-Clenshaw A^{-1/4} of degree `degree` on [lo, hi]."""
    lib = load_library()
    n, b, X = _root_common(A, scale, X)
    p = _prec(prec)
    if ws is None:
        ws = workspace(OP_INV_ROOT_CHEB, n, b, p, degree, device=A.device)
    _check(lib.inv_root_cheb(_ptr(A), float(ridge), _ptr(scale), n, b, int(degree), float(lo),
                             float(hi), p, _ptr(X), _ptr(ws), _nbytes(ws), _stream()),
           "inv_root_cheb")
    return X


def precondition_apply(G, Froot, prec=FP32_3XTF32, U=None, ws=None):
    """U_j = Froot[j] G_j Froot[Ng + j]."""
    lib = load_library()
    _stack(G, "G", G.dtype)
    ng, b = _blocks3(G, "G")
    _shape(_stack(Froot, "Froot"), (2 * ng, b, b), "Froot")
    p = _prec(prec)
    if U is None:
        U = torch.empty((ng, b, b), dtype=torch.float32, device=G.device)
    _shape(_stack(U, "U"), (ng, b, b), "U")
    if ws is None:
        ws = workspace(OP_PRECONDITION_APPLY, ng, b, p, device=G.device)
    _check(lib.precondition_apply(_ptr(G), _gdt(G), _ptr(Froot), ng, b, p, _ptr(U), _ptr(ws),
                                  _nbytes(ws), _stream()), "precondition_apply")
    return U


def precondition_update(G, Froot, W, lr, prec=FP32_3XTF32, U=None, ws=None):
    """W_j -= lr * Froot[j] G_j Froot[Ng + j], in place on W (Ng, B, B) fp32; U optional."""
    lib = load_library()
    _stack(G, "G", G.dtype)
    ng, b = _blocks3(G, "G")
    _shape(_stack(Froot, "Froot"), (2 * ng, b, b), "Froot")
    _shape(_stack(W, "W"), (ng, b, b), "W")
    p = _prec(prec)
    if U is not None:
        _shape(_stack(U, "U"), (ng, b, b), "U")
    if ws is None:
        ws = workspace(OP_PRECONDITION_APPLY, ng, b, p, device=G.device)
    _check(lib.precondition_update(_ptr(G), _gdt(G), _ptr(Froot), ng, b, p, float(lr), _ptr(W),
                                   _ptr(U), _ptr(ws), _nbytes(ws), _stream()),
           "precondition_update")
    return W


def _matrix(M, name):
    if not isinstance(M, torch.Tensor) or not M.is_cuda or M.dim() != 2:
        raise TypeError("%s must be a 2-D CUDA tensor" % name)
    if M.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)
    return M


def pack_blocks(M, B, out=None, valid=True):
    """Row-block-major (ceil(rows/B) * ceil(cols/B), B, B) blocks of the 2-D matrix M,
    zero-padded; returns (blocks, valid_rows, valid_cols) (the last two None if
    valid is False).  M may be a row-strided view."""
    lib = load_library()
    _matrix(M, "M")
    rows, cols = M.shape
    nb = -(-rows // B) * -(-cols // B)
    if out is None:
        out = torch.empty((nb, B, B), dtype=M.dtype, device=M.device)
    _shape(_stack(out, "out", M.dtype), (nb, B, B), "out")
    vr = torch.empty(nb, dtype=torch.int32, device=M.device) if valid else None
    vc = torch.empty(nb, dtype=torch.int32, device=M.device) if valid else None
    _check(lib.pack_blocks(_ptr(M), _gdt(M), rows, cols, M.stride(0), B, _ptr(out), _ptr(vr),
                           _ptr(vc), _stream()), "pack_blocks")
    return out, vr, vc


def unpack_blocks(blocks, rows, cols, out=None):
    """The (rows, cols) matrix whose row-block-major blocks are `blocks` (padding
    dropped); `out` may be a row-strided 2-D view."""
    lib = load_library()
    _stack(blocks, "blocks", blocks.dtype)
    _, B = _blocks3(blocks, "blocks")
    nb = -(-rows // B) * -(-cols // B)
    if blocks.shape[0] < nb:
        raise ValueError("blocks holds %d blocks, a (%d, %d) matrix needs %d"
                         % (blocks.shape[0], rows, cols, nb))
    if out is None:
        out = torch.empty((rows, cols), dtype=blocks.dtype, device=blocks.device)
    _matrix(out, "out")
    if out.dtype != blocks.dtype or tuple(out.shape) != (rows, cols):
        raise ValueError("out must be (rows, cols) of the blocks' dtype")
    _check(lib.unpack_blocks(_ptr(blocks), _gdt(blocks), rows, cols, out.stride(0), B, _ptr(out),
                             _stream()), "unpack_blocks")
    return out


def gemm(A, B, prec=TF32, trans_a=False, trans_b=False, A_lo=None, B_lo=None, C=None):
    """C[k] = op(A[k]) op(B[k]) on the tensor cores; operands already in prec's format."""
    lib = load_library()
    p = _prec(prec)
    _stack(A, "A", A.dtype)
    n, b = _blocks3(A, "A")
    _shape(_stack(B, "B", A.dtype), (n, b, b), "B")
    for t, name in ((A_lo, "A_lo"), (B_lo, "B_lo")):
        if t is not None:
            _shape(_stack(t, name, A.dtype), (n, b, b), name)
    if C is None:
        C = torch.empty((n, b, b), dtype=torch.float32, device=A.device)
    _shape(_stack(C, "C"), (n, b, b), "C")
    _check(lib.dash_gemm(_ptr(A), _ptr(A_lo), int(bool(trans_a)), _ptr(B), _ptr(B_lo),
                         int(bool(trans_b)), n, b, p, _ptr(C), _stream()), "dash_gemm")
    return C


def gemm_ex(A, B, prec=TF32, sym=0, trans_a=False, trans_b=False, A_lo=None, B_lo=None, C=None):
    """dash_gemm_ex: symmetric-half operand forms (sym 1-4: 1 both operands read from
    their upper 256-tiles, 2 as 1 with only C's upper tiles written, 3 whole operands
    with only C's upper tiles written, 4 only A read from its upper tiles) and, for
    16-bit prec, a 16-bit pair B (B_lo given): C = A B + A B_lo."""
    lib = load_library()
    p = _prec(prec)
    _stack(A, "A", A.dtype)
    n, b = _blocks3(A, "A")
    _shape(_stack(B, "B", A.dtype), (n, b, b), "B")
    for t, name in ((A_lo, "A_lo"), (B_lo, "B_lo")):
        if t is not None:
            _shape(_stack(t, name, A.dtype), (n, b, b), name)
    if C is None:
        C = torch.empty((n, b, b), dtype=torch.float32, device=A.device)
    _shape(_stack(C, "C"), (n, b, b), "C")
    _check(lib.dash_gemm_ex(_ptr(A), _ptr(A_lo), int(bool(trans_a)), _ptr(B), _ptr(B_lo),
                            int(bool(trans_b)), n, b, p, int(sym), _ptr(C), _stream()),
           "dash_gemm_ex")
    return C
