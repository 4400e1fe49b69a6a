"""Thin Python binding of libdas (ctypes; argument marshalling only).

Every step of the computation runs in the CUDA library: this module only
loads ``_lib/libdas.so``, checks tensor arguments and forwards raw pointers and
the current torch stream.  There is no fallback: if the library is missing the
import of :func:`lib` raises, so a GPU path can never silently run elsewhere.

Names follow the C ABI in ``include/das.h``: :class:`Plan` wraps
``das_plan_create`` / ``das_beamform`` / ``das_plan_destroy``, :func:`permute`
wraps ``das_permute``.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

LIBRARY = Path(__file__).resolve().parent / "_lib" / "libdas.so"

DAS_OK, DAS_ERR_INVALID_ARG, DAS_ERR_UNSUPPORTED, DAS_ERR_OUT_OF_MEMORY, DAS_ERR_CUDA, \
    DAS_ERR_TIMEOUT = range(6)
DAS_F32, DAS_C64, DAS_F64, DAS_C128, DAS_F16, DAS_C32H = 0, 1, 2, 3, 4, 5
_DTYPES = {"f32": DAS_F32, "c64": DAS_C64, "f64": DAS_F64, "c128": DAS_C128, "f16": DAS_F16,
           "c32h": DAS_C32H}
KERNELS = {"auto": 0, "bl": 1, "bi": 2, "brick": 3, "window": 4, "pair": 5}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}
OPT_KERNEL, OPT_DEMOD_HZ, OPT_TIMING, OPT_BI_GROUP, OPT_HOST_GROUPS, OPT_STORAGE, OPT_RX_GROUPS, \
    OPT_TX_GROUPS = 0, 1, 2, 3, 4, 5, 6, 7
STORAGE_NATIVE, STORAGE_F16 = 0, 1

# every function the header declares, with its ctypes signature
_VP = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SIGS = {
    "das_plan_create": (_I, [ctypes.POINTER(_VP), _VP, _VP, _F, _F, _F, _F, _I, _I, _I, _I, _I]),
    "das_plan_create_points": (_I, [ctypes.POINTER(_VP), _VP, _I, _VP, _F, _F, _F, _F, _I, _I, _I, _I, _I]),
    "das_plan_set_option": (_I, [_VP, _I, ctypes.c_double]),
    "das_plan_get_option": (_I, [_VP, _I, ctypes.POINTER(ctypes.c_double)]),
    "das_plan_kernel": (_I, [_VP, ctypes.POINTER(_I)]),
    "das_plan_launches": (_I, [_VP, ctypes.POINTER(_I)]),
    "das_beamform": (_I, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "das_beamform_host": (_I, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "das_beamform_host_volumes": (_I, [_VP, _I, _VP, _VP, _VP, _VP, _VP]),
    "das_plan_last_times": (_I, [_VP, ctypes.POINTER(_F), ctypes.POINTER(_F)]),
    "das_plan_device_bytes": (_I, [_VP, ctypes.POINTER(ctypes.c_size_t)]),
    "das_plan_destroy": (_I, [_VP]),
    "das_permute": (_I, [_VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "das_permute_bqmk_to_kqmb": (_I, [_VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "das_beamform_noalloc": (_I, [_VP, _VP, _F, _F, _F, _F, ctypes.c_double, _I, _I, _I, _I, _I,
                                  _VP, _VP, _VP, _VP, _VP]),
    "das_last_error_string": (ctypes.c_char_p, []),
    "das_version": (ctypes.c_char_p, []),
}


class DasError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libdas error {status}: {message}")
        self.status = status


class _Grid(ctypes.Structure):
    _fields_ = [("nx", _I), ("ny", _I), ("nz", _I),
                ("x0", _F), ("y0", _F), ("z0", _F), ("dx", _F), ("dy", _F), ("dz", _F),
                ("xyz", ctypes.c_void_p)]


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libdas (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not LIBRARY.exists():
            raise ImportError(f"libdas.so not built ({LIBRARY}); run __graft_entry__.build()")
        h = ctypes.CDLL(str(LIBRARY))
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = h
    return _LIB


def _check(status: int):
    if status != DAS_OK:
        raise DasError(status, lib().das_last_error_string().decode())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, name, dtype=None, numel=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


class Plan:
    """A DAS plan: fixed grid, receivers, physics constants, dtype and sizes."""

    def __init__(self, grid, rx_xyz, c, fs, t0=0.0, fnum=0.0, dtype="f32", B=1, Q=1, M=None,
                 K=1, kernel="auto", f_demod=0.0, storage="native", points=None):
        """``grid`` = (nx, ny, nz, x0, y0, z0, dx, dy, dz), or None with ``points``
        an N x 3 array of voxel positions (das_plan_create_points).  With both,
        ``points`` (nx*ny*nz x 3) goes in the grid's voxel list (das_plan_create
        with grid.xyz)."""
        rx = np.ascontiguousarray(rx_xyz, dtype=np.float32).reshape(-1, 3)
        M = rx.shape[0] if M is None else M
        if M != rx.shape[0]:
            raise ValueError("M does not match rx_xyz")
        self.dtype = dtype
        self.B, self.Q, self.M, self.K = int(B), int(Q), int(M), int(K)
        h = ctypes.c_void_p()
        dt = _DTYPES[dtype]
        self._rx = rx
        if points is not None and grid is not None:
            pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 3)
            self.grid = None
            self.N = int(grid[0]) * int(grid[1]) * int(grid[2])
            if pts.shape[0] != self.N:
                raise ValueError("points must hold nx*ny*nz positions")
            g = _Grid(*[int(v) for v in grid[:3]], *[float(v) for v in tuple(grid)[3:9]],
                      pts.ctypes.data_as(ctypes.c_void_p))
            _check(lib().das_plan_create(ctypes.byref(h), ctypes.byref(g),
                                         rx.ctypes.data_as(ctypes.c_void_p), c, fs, t0, fnum, dt,
                                         self.B, self.Q, self.M, self.K))
        elif points is not None:
            pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 3)
            self.grid = None
            self.N = pts.shape[0]
            _check(lib().das_plan_create_points(
                ctypes.byref(h), pts.ctypes.data_as(ctypes.c_void_p), self.N,
                rx.ctypes.data_as(ctypes.c_void_p), c, fs, t0, fnum, dt, self.B, self.Q, self.M,
                self.K))
        else:
            self.grid = tuple(grid)
            self.N = self.grid[0] * self.grid[1] * self.grid[2]
            g = _Grid(*[int(v) for v in self.grid[:3]], *[float(v) for v in self.grid[3:]])
            _check(lib().das_plan_create(ctypes.byref(h), ctypes.byref(g),
                                         rx.ctypes.data_as(ctypes.c_void_p), c, fs, t0, fnum, dt,
                                         self.B, self.Q, self.M, self.K))
        self._h = h
        if kernel != "auto":
            self.set_option(OPT_KERNEL, KERNELS[kernel])
        if f_demod:
            self.set_option(OPT_DEMOD_HZ, f_demod)
        if storage != "native":
            self.set_option(OPT_STORAGE, {"native": STORAGE_NATIVE, "f16": STORAGE_F16}[storage])

    # -- options
    def set_option(self, opt: int, value: float):
        _check(lib().das_plan_set_option(self._h, opt, float(value)))

    def get_option(self, opt: int) -> float:
        v = ctypes.c_double()
        _check(lib().das_plan_get_option(self._h, opt, ctypes.byref(v)))
        return v.value

    @property
    def kernel(self) -> str:
        k = ctypes.c_int()
        _check(lib().das_plan_kernel(self._h, ctypes.byref(k)))
        return KERNEL_NAMES[k.value]

    @kernel.setter
    def kernel(self, name: str):
        self.set_option(OPT_KERNEL, KERNELS[name])

    @property
    def launches(self) -> int:
        """Kernel launches one beamform call makes with the current options."""
        n = ctypes.c_int()
        _check(lib().das_plan_launches(self._h, ctypes.byref(n)))
        return n.value

    # -- compute
    def _torch_dtypes(self):
        """(float32, record dtype, output dtype): half records give float32 /
        complex64 output."""
        import torch
        rec = {"f32": torch.float32, "c64": torch.complex64, "f64": torch.float64,
               "c128": torch.complex128, "f16": torch.float16, "c32h": torch.complex32}[self.dtype]
        outd = {"f16": torch.float32, "c32h": torch.complex64}.get(self.dtype, rec)
        return torch.float32, rec, outd

    def beamform(self, rf, tau_tx, w_tx, out=None, stream=None):
        """y (B x N) from device tensors rf (B x Q x M x K), tau_tx / w_tx (Q x N)."""
        import torch
        f32, el, el_out = self._torch_dtypes()
        if out is None:
            out = torch.empty((self.B, self.N), dtype=el_out, device=rf.device)
        _check(lib().das_beamform(
            self._h, _dev_ptr(rf, "rf", el, self.B * self.Q * self.M * self.K),
            _dev_ptr(tau_tx, "tau_tx", f32, self.Q * self.N), _dev_ptr(w_tx, "w_tx", f32, self.Q * self.N),
            _dev_ptr(out, "out", el_out, self.B * self.N), _stream_handle(stream)))
        return out

    def beamform_host(self, rf, tau_tx, w_tx, out, stream=None):
        """Same computation from host arrays/tensors (copies inside, synchronous)."""
        def hp(a, name, n):
            import torch
            if isinstance(a, torch.Tensor):
                if a.is_cuda or not a.is_contiguous() or a.numel() != n:
                    raise ValueError(f"{name} must be a contiguous host tensor of {n} elements")
                return ctypes.c_void_p(a.data_ptr())
            if not (isinstance(a, np.ndarray) and a.flags.c_contiguous and a.size == n):
                raise ValueError(f"{name} must be a contiguous host array of {n} elements")
            return a.ctypes.data_as(ctypes.c_void_p)
        _check(lib().das_beamform_host(
            self._h, hp(rf, "rf", self.B * self.Q * self.M * self.K),
            hp(tau_tx, "tau_tx", self.Q * self.N), hp(w_tx, "w_tx", self.Q * self.N),
            hp(out, "out", self.B * self.N), _stream_handle(stream)))
        return out

    def beamform_host_volumes(self, rf, tau_tx, w_tx, out, stream=None):
        """A stream of V volumes from host memory: rf V x B x Q x M x K, out
        V x B x N, one tau_tx / w_tx (Q x N) for all (copies inside, synchronous)."""
        import torch
        n_rec = self.B * self.Q * self.M * self.K
        def host(a, name):
            if isinstance(a, torch.Tensor):
                if a.is_cuda or not a.is_contiguous():
                    raise ValueError(f"{name} must be a contiguous host tensor")
                return a.numel(), ctypes.c_void_p(a.data_ptr())
            if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
                raise ValueError(f"{name} must be a contiguous host array")
            return a.size, a.ctypes.data_as(ctypes.c_void_p)
        n_rf, p_rf = host(rf, "rf")
        if n_rf % n_rec != 0 or n_rf == 0:
            raise ValueError(f"rf must hold a whole number of {n_rec}-element records")
        vols = n_rf // n_rec
        n_out, p_out = host(out, "out")
        if n_out != vols * self.B * self.N:
            raise ValueError(f"out must hold {vols} x {self.B} x {self.N} elements")
        n_t, p_t = host(tau_tx, "tau_tx")
        n_w, p_w = host(w_tx, "w_tx")
        if n_t != self.Q * self.N or n_w != self.Q * self.N:
            raise ValueError("tau_tx and w_tx must hold Q x N elements")
        _check(lib().das_beamform_host_volumes(self._h, vols, p_rf, p_t, p_w, p_out, _stream_handle(stream)))
        return out

    def last_times(self):
        """(permute_ms, das_ms) of the last beamform when timing is on."""
        a, b = ctypes.c_float(), ctypes.c_float()
        _check(lib().das_plan_last_times(self._h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def device_bytes(self) -> int:
        v = ctypes.c_size_t()
        _check(lib().das_plan_device_bytes(self._h, ctypes.byref(v)))
        return v.value

    def close(self):
        if getattr(self, "_h", None):
            _check(lib().das_plan_destroy(self._h))
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def permute(rf, out, layout: int = 0, stream=None, storage: str = "native"):
    """B x Q x M x K -> K x Q x M x B (layout 0), Q x M x K x B (layout 1),
    Q x M x (K+3) x B with sample k at row k + 1 and pad rows untouched (layout 2)
    or (K+2) x Q x M x B with sample k at plane k + 1 and pad planes untouched
    (layout 3).
    ``storage="native"`` copies bit for bit; ``"f16"`` writes float16 (float32 data)
    or complex32 as pairs of float16 (complex64 data), ``out`` being a float16
    tensor with 1 or 2 values per element.  float16 and complex32 records are
    copied bit for bit either way (``out`` of the record's dtype)."""
    import torch
    dts = {torch.float32: DAS_F32, torch.complex64: DAS_C64, torch.float16: DAS_F16,
           torch.complex32: DAS_C32H}
    if rf.dtype not in dts or rf.dim() != 4:
        raise TypeError("rf must be a 4-D float32, complex64, float16 or complex32 CUDA tensor")
    B, Q, M, K = rf.shape
    dt = dts[rf.dtype]
    n_out = B * Q * M * (K + {2: 3, 3: 2}.get(layout, 0))
    if storage == "f16" and dt in (DAS_F32, DAS_C64):
        n_out *= 2 if dt == DAS_C64 else 1
        optr = _dev_ptr(out, "out", torch.float16, n_out)
    else:
        optr = _dev_ptr(out, "out", rf.dtype, n_out)
    st = {"native": STORAGE_NATIVE, "f16": STORAGE_F16}[storage]
    _check(lib().das_permute(_dev_ptr(rf, "rf"), optr, dt, B, Q, M, K, layout, st,
                             _stream_handle(stream)))
    return out


def permute_bqmk_to_kqmb(rf, out, stream=None):
    """das_permute_bqmk_to_kqmb: B x Q x M x K -> K x Q x M x B, bit for bit."""
    import torch
    if rf.dtype not in (torch.float32, torch.complex64) or rf.dim() != 4:
        raise TypeError("rf must be a 4-D float32 or complex64 CUDA tensor")
    B, Q, M, K = rf.shape
    dt = DAS_C64 if rf.dtype == torch.complex64 else DAS_F32
    _check(lib().das_permute_bqmk_to_kqmb(_dev_ptr(rf, "rf"), _dev_ptr(out, "out", rf.dtype, B * Q * M * K),
                                          dt, B, Q, M, K, _stream_handle(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 64 << 20


def beamform_noalloc(grid, rx_xyz, c, fs, t0, fnum, f_demod, rf, tau_tx, w_tx, out,
                     stream=None):
    """das_beamform_noalloc: the brick-kernel beamform without any device
    allocation, for callers that cannot call cudaMalloc while they run (its
    scratch is a 64 MiB static array inside libdas; see include/das.h).
    ``rx_xyz`` is a CUDA tensor (M x 3 float32); rf (B x Q x M x K), tau_tx and
    w_tx (Q x N) and out (B x N) are CUDA tensors as for :meth:`Plan.beamform`."""
    import torch
    B, Q, M, K = rf.shape
    dt = DAS_C64 if rf.dtype == torch.complex64 else DAS_F32
    N = int(grid[0]) * int(grid[1]) * int(grid[2])
    g = _Grid(*[int(v) for v in grid[:3]], *[float(v) for v in grid[3:]])
    _check(lib().das_beamform_noalloc(
        ctypes.byref(g), _dev_ptr(rx_xyz, "rx_xyz", torch.float32, M * 3), c, fs, t0, fnum,
        float(f_demod), dt, B, Q, M, K, _dev_ptr(rf, "rf", rf.dtype),
        _dev_ptr(tau_tx, "tau_tx", torch.float32, Q * N), _dev_ptr(w_tx, "w_tx", torch.float32, Q * N),
        _dev_ptr(out, "out", rf.dtype, B * N), _stream_handle(stream)))
    return out
