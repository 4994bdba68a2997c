"""Python binding of liblopt (include/lopt.h): argument marshalling only.

Every step of the optimizer runs inside the library's CUDA kernels; this
module converts torch tensors to device pointers and calls the C ABI.  There
is no fallback: if liblopt.so is missing or a tensor is not a contiguous
CUDA float32 tensor, the call raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblopt.so")

LOPT_OK = 0
LOPT_D_FEAT = 39
LOPT_N_STATS = 28
MLP_FP32 = 0
MLP_TC = 1
_PATHS = {"fp32": MLP_FP32, "tc": MLP_TC}

ERRORS = {
    -1: "LOPT_E_ARG", -2: "LOPT_E_SHAPE", -3: "LOPT_E_ALIGN", -4: "LOPT_E_CUDA",
    -5: "LOPT_E_OOM", -6: "LOPT_E_UNSUPPORTED", -7: "LOPT_E_TIMEOUT", -8: "LOPT_E_ALIAS",
    -9: "LOPT_E_TOO_LARGE",
}

EXPORTED = ("lopt_weight_set_size", "lopt_create", "lopt_set_mlp_path", "lopt_set_weight_decay",
            "lopt_set_sweep_bytes", "lopt_step",
            "lopt_step_host", "lopt_host_sync", "lopt_set_host_groups",
            "lopt_shard_sizes", "lopt_shard_begin", "lopt_shard_middle", "lopt_shard_end",
            "lopt_schedule_info", "lopt_check", "lopt_feature_stats", "lopt_set_kernel_timing", "lopt_kernel_times",
            "lopt_rowcol_static", "lopt_selftest_wait", "lopt_destroy", "lopt_strerror", "lopt_last_cuda_error",
            "lopt_version")


class LoptTensor(ctypes.Structure):
    """Mirror of lopt_tensor."""
    _fields_ = [
        ("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
        ("mom", ctypes.c_void_p * 3), ("rms", ctypes.c_void_p),
        ("row", ctypes.c_void_p * 3), ("col", ctypes.c_void_p * 3),
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
        ("weight_set", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


class LoptError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__("%s failed: %s (%s, %d)" % (fn, msg, ERRORS.get(code, "?"), code))
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblopt.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("liblopt.so not found at %s; build it with "
                          "learned_optimizer_step_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.lopt_weight_set_size.argtypes = [i32, i32]
    lib.lopt_weight_set_size.restype = i32
    lib.lopt_create.argtypes = [ctypes.POINTER(ctypes.c_float), i32, i32, i32, ctypes.POINTER(vp)]
    lib.lopt_create.restype = i32
    lib.lopt_set_mlp_path.argtypes = [vp, i32]
    lib.lopt_set_mlp_path.restype = i32
    lib.lopt_set_weight_decay.argtypes = [vp, ctypes.c_float]
    lib.lopt_set_weight_decay.restype = i32
    lib.lopt_set_sweep_bytes.argtypes = [vp, i64]
    lib.lopt_set_sweep_bytes.restype = i32
    lib.lopt_selftest_wait.argtypes = [i64]
    lib.lopt_selftest_wait.restype = i32
    lib.lopt_step.argtypes = [vp, ctypes.POINTER(LoptTensor), i32, i64, ctypes.c_float, vp]
    lib.lopt_step_host.restype = i32
    lib.lopt_step_host.argtypes = [vp, ctypes.POINTER(LoptTensor), i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                   i64, ctypes.c_float, vp]
    lib.lopt_host_sync.restype = i32
    lib.lopt_host_sync.argtypes = [vp, vp]
    lib.lopt_set_host_groups.restype = i32
    lib.lopt_set_host_groups.argtypes = [vp, i32]
    lib.lopt_step.restype = i32
    lib.lopt_shard_sizes.argtypes = [ctypes.POINTER(LoptTensor), i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.lopt_shard_sizes.restype = i32
    lib.lopt_shard_begin.argtypes = [vp, ctypes.POINTER(LoptTensor), ctypes.POINTER(i64), i32, i64, ctypes.c_float,
                                     vp, vp, vp]
    lib.lopt_shard_begin.restype = i32
    p32 = ctypes.POINTER(ctypes.c_int32)
    lib.lopt_schedule_info.argtypes = [ctypes.POINTER(LoptTensor), i32, i64, p32, p32, p32, p32, p32]
    lib.lopt_schedule_info.restype = i32
    lib.lopt_shard_middle.argtypes = [vp, vp]
    lib.lopt_shard_middle.restype = i32
    lib.lopt_shard_end.argtypes = [vp, vp]
    lib.lopt_shard_end.restype = i32
    lib.lopt_check.argtypes = [vp]
    lib.lopt_check.restype = i32
    lib.lopt_feature_stats.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_double)]
    lib.lopt_feature_stats.restype = i32
    lib.lopt_set_kernel_timing.argtypes = [vp, i32]
    lib.lopt_set_kernel_timing.restype = i32
    lib.lopt_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    lib.lopt_kernel_times.restype = i32
    lib.lopt_rowcol_static.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i64, i64, vp, vp]
    lib.lopt_rowcol_static.restype = i32
    lib.lopt_destroy.argtypes = [vp]
    lib.lopt_destroy.restype = i32
    lib.lopt_strerror.argtypes = [i32]
    lib.lopt_last_cuda_error.restype = ctypes.c_char_p
    lib.lopt_last_cuda_error.argtypes = []
    lib.lopt_strerror.restype = ctypes.c_char_p
    lib.lopt_version.argtypes = []
    lib.lopt_version.restype = i32
    _lib = lib
    return lib


def schedule_info(shapes, sweep_bytes: int = 0) -> dict:
    """The launch schedule lopt_step builds for tensors of these [rows x
    cols] views (host only, no device): per kernel (K0 row strips, K1 and
    K2 element chunks) the units in launch order as [n x 2] int32 arrays of
    (tensor, index within the tensor); the rows of each tensor's K0 strips;
    and the single-sweep groups as [g x 6] (first unit and count of K0, K1,
    K2)."""
    import numpy as np
    lib = load_library()
    n = len(shapes)
    arr = (LoptTensor * max(n, 1))()
    for i, (r, c) in enumerate(shapes):
        arr[i].rows, arr[i].cols = int(r), int(c)
    n_units = (ctypes.c_int32 * 3)()
    n_groups = ctypes.c_int32()
    _check("lopt_schedule_info", lib.lopt_schedule_info(arr, n, int(sweep_bytes), n_units, None, None,
                                                        ctypes.byref(n_groups), None))
    counts = [int(x) for x in n_units]
    units = np.zeros((sum(counts), 2), dtype=np.int32)
    strips = np.zeros(max(n, 1), dtype=np.int32)
    groups = np.zeros((max(n_groups.value, 1), 6), dtype=np.int32)
    as_p32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    _check("lopt_schedule_info", lib.lopt_schedule_info(arr, n, int(sweep_bytes), n_units, as_p32(units),
                                                        as_p32(strips), ctypes.byref(n_groups), as_p32(groups)))
    a, b = counts[0], counts[0] + counts[1]
    return {"k0": units[:a], "k1": units[a:b], "k2": units[b:], "strip_rows": strips[:n],
            "groups": groups[:n_groups.value]}


def _check(fn: str, code: int) -> None:
    if code != LOPT_OK:
        lib = load_library()
        msg = lib.lopt_strerror(code).decode()
        if code in (-4, -5):   # LOPT_E_CUDA, LOPT_E_OOM: name the CUDA error
            msg += " [%s]" % lib.lopt_last_cuda_error().decode()
        raise LoptError(fn, code, msg)


def _ptr(t, n: int, what: str) -> int:
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA float32 tensor" % what)
    if t.numel() != n:
        raise ValueError("%s has %d elements, expected %d" % (what, t.numel(), n))
    return t.data_ptr()


def _host_ptr(t, n: int, what: str) -> int:
    """Address of a CPU float32 buffer of n elements (torch tensor or numpy array)."""
    import torch
    if isinstance(t, np.ndarray):
        if t.dtype != np.float32 or not t.flags["C_CONTIGUOUS"] or not t.flags["WRITEABLE"]:
            raise TypeError("%s must be a writeable contiguous float32 array" % what)
        if t.size != n:
            raise ValueError("%s has %d elements, expected %d" % (what, t.size, n))
        return t.ctypes.data
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor or a numpy array" % what)
    if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CPU float32 tensor" % what)
    if t.numel() != n:
        raise ValueError("%s has %d elements, expected %d" % (what, t.numel(), n))
    return t.data_ptr()


@dataclass
class TensorState:
    """One parameter tensor and its optimizer state (all CUDA float32)."""
    param: "object"
    grad: "object"
    mom: List["object"]
    rms: "object"
    row: List["object"]
    col: List["object"]
    rows: int
    cols: int
    weight_set: int = 0

    @staticmethod
    def from_dict(d: dict) -> "TensorState":
        return TensorState(d["param"], d["grad"], list(d["mom"]), d["rms"], list(d["row"]),
                           list(d["col"]), int(d["rows"]), int(d["cols"]), int(d.get("weight_set", 0)))

    def to_c(self) -> LoptTensor:
        n = self.rows * self.cols
        c = LoptTensor()
        c.param = _ptr(self.param, n, "param")
        c.grad = _ptr(self.grad, n, "grad")
        for k in range(3):
            c.mom[k] = _ptr(self.mom[k], n, "mom[%d]" % k)
            c.row[k] = _ptr(self.row[k], self.rows, "row[%d]" % k)
            c.col[k] = _ptr(self.col[k], self.cols, "col[%d]" % k)
        c.rms = _ptr(self.rms, n, "rms")
        c.rows, c.cols, c.weight_set, c.reserved = self.rows, self.cols, self.weight_set, 0
        return c


class PreparedList:
    """A parameter list marshalled once into the C descriptor array."""

    def __init__(self, tensors: Sequence[TensorState]):
        self.tensors = list(tensors)
        self.array = (LoptTensor * len(self.tensors))(*[t.to_c() for t in self.tensors])
        self.n = len(self.tensors)
        self.numel = sum(t.rows * t.cols for t in self.tensors)


def weight_set_size(hidden: int) -> int:
    n = load_library().lopt_weight_set_size(LOPT_D_FEAT, int(hidden))
    if n < 0:
        _check("lopt_weight_set_size", n)
    return n


class LearnedOptimizer:
    """One library handle: MLP weight sets + workspace.  ``step`` runs one
    learned-optimizer step over a whole parameter list."""

    def __init__(self, weights: np.ndarray, hidden: int = 32, mlp_path: str = "fp32"):
        lib = load_library()
        w = np.ascontiguousarray(np.asarray(weights, dtype=np.float32))
        size = weight_set_size(hidden)
        if w.size % size != 0 or w.size == 0:
            raise ValueError("weights must hold n_sets * %d floats" % size)
        self.hidden = int(hidden)
        self.n_sets = w.size // size
        self._w = w
        h = ctypes.c_void_p()
        _check("lopt_create", lib.lopt_create(w.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                              LOPT_D_FEAT, self.hidden, self.n_sets, ctypes.byref(h)))
        self._h = h
        self.set_mlp_path(mlp_path)

    def set_mlp_path(self, path: str) -> None:
        _check("lopt_set_mlp_path", load_library().lopt_set_mlp_path(self._h, _PATHS[path]))
        self.mlp_path = path

    def set_weight_decay(self, weight_decay: float) -> None:
        """Decoupled weight decay of later steps: p -= lr * (update + wd * p)."""
        _check("lopt_set_weight_decay", load_library().lopt_set_weight_decay(self._h, float(weight_decay)))

    def set_sweep_bytes(self, group_bytes: int) -> None:
        """Groups of consecutive tensors with at most ``group_bytes`` of state
        (24 bytes per element) run the three kernels one group after the
        other, so that re-reads come from L2; 0 turns it off."""
        _check("lopt_set_sweep_bytes", load_library().lopt_set_sweep_bytes(self._h, int(group_bytes)))

    def prepare(self, tensors: Sequence) -> PreparedList:
        ts = [t if isinstance(t, TensorState) else TensorState.from_dict(t) for t in tensors]
        return PreparedList(ts)

    def step(self, tensors, t: int, lr: float = 1.0, stream: Optional[object] = None) -> None:
        """Enqueue one step (asynchronous on ``stream``; default: torch's
        current stream)."""
        import torch
        pl = tensors if isinstance(tensors, PreparedList) else self.prepare(tensors)
        if stream is None:
            stream = torch.cuda.current_stream()
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        _check("lopt_step", load_library().lopt_step(self._h, pl.array, pl.n, int(t), float(lr),
                                                      ctypes.c_void_p(handle)))

    def step_host(self, tensors, grad_host, param_host, t: int, lr: float = 1.0,
                  stream: Optional[object] = None) -> None:
        """One step with gradients coming from and parameters going to host
        memory: grad_host[i] is tensor i's gradient (its device ``grad`` is
        not used) and the new parameters are copied into param_host[i] (CPU
        float32 buffers of rows * cols elements; pinned memory lets the
        copies overlap the kernels).  The kernels are asynchronous on
        ``stream``; the parameter copies may still run after it: call
        ``host_sync`` (or ``check``) before reading param_host or refilling
        grad_host."""
        pl = tensors if isinstance(tensors, PreparedList) else self.prepare(tensors)
        if len(grad_host) != pl.n or len(param_host) != pl.n:
            raise ValueError("one host gradient and one host parameter buffer per tensor")
        gp = (ctypes.c_void_p * pl.n)(*[_host_ptr(x, ts.rows * ts.cols, "grad_host[%d]" % i)
                                        for i, (x, ts) in enumerate(zip(grad_host, pl.tensors))])
        pp = (ctypes.c_void_p * pl.n)(*[_host_ptr(x, ts.rows * ts.cols, "param_host[%d]" % i)
                                        for i, (x, ts) in enumerate(zip(param_host, pl.tensors))])
        _check("lopt_step_host", load_library().lopt_step_host(self._h, pl.array, pl.n, gp, pp, int(t), float(lr),
                                                                self._stream(stream)))

    def set_host_groups(self, max_groups: int) -> None:
        """Most groups of tensors a host-buffer step uses (1..16; default 2)."""
        _check("lopt_set_host_groups", load_library().lopt_set_host_groups(self._h, int(max_groups)))

    def host_sync(self, stream: Optional[object] = None) -> None:
        """Make ``stream`` wait for every parameter copy of the host-buffer
        steps enqueued so far."""
        _check("lopt_host_sync", load_library().lopt_host_sync(self._h, self._stream(stream)))

    # ---- row-sharded step --------------------------------------------------
    @staticmethod
    def shard_buffers(tensors, device=None):
        """Exchange buffers (float64, on the GPU) of a row-sharded step."""
        import torch
        pl = tensors if isinstance(tensors, PreparedList) else PreparedList(
            [t if isinstance(t, TensorState) else TensorState.from_dict(t) for t in tensors])
        n1, n2 = ctypes.c_int64(), ctypes.c_int64()
        _check("lopt_shard_sizes", load_library().lopt_shard_sizes(pl.array, pl.n, ctypes.byref(n1),
                                                                    ctypes.byref(n2)))
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        return (torch.zeros(n1.value, dtype=torch.float64, device=dev),
                torch.zeros(n2.value, dtype=torch.float64, device=dev))

    @staticmethod
    def _stream(stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))

    def shard_begin(self, tensors, global_rows, t: int, lr: float, x1, x2, stream=None) -> None:
        pl = tensors if isinstance(tensors, PreparedList) else self.prepare(tensors)
        gr = (ctypes.c_int64 * pl.n)(*[int(r) for r in global_rows])
        for x in (x1, x2):
            if not x.is_cuda or x.dtype.itemsize != 8 or not x.is_contiguous():
                raise TypeError("exchange buffers must be contiguous CUDA float64 tensors")
        _check("lopt_shard_begin", load_library().lopt_shard_begin(
            self._h, pl.array, gr, pl.n, int(t), float(lr), ctypes.c_void_p(x1.data_ptr()),
            ctypes.c_void_p(x2.data_ptr()), self._stream(stream)))

    def shard_middle(self, stream=None) -> None:
        _check("lopt_shard_middle", load_library().lopt_shard_middle(self._h, self._stream(stream)))

    def shard_end(self, stream=None) -> None:
        _check("lopt_shard_end", load_library().lopt_shard_end(self._h, self._stream(stream)))

    def sharded_step(self, tensors, global_rows, t: int, lr: float, x1, x2, all_reduce,
                     stream=None) -> None:
        """One row-sharded step; ``all_reduce(buffer)`` sums a float64 CUDA
        buffer over the ranks in place (e.g. torch.distributed.all_reduce)."""
        self.shard_begin(tensors, global_rows, t, lr, x1, x2, stream)
        all_reduce(x1)
        self.shard_middle(stream)
        all_reduce(x2)
        self.shard_end(stream)

    def check(self) -> None:
        """Wait for the last step; raise if a kernel reported an error."""
        _check("lopt_check", load_library().lopt_check(self._h))

    def feature_stats(self, index: int) -> np.ndarray:
        out = np.zeros(LOPT_N_STATS, dtype=np.float64)
        _check("lopt_feature_stats", load_library().lopt_feature_stats(
            self._h, int(index), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))))
        return out

    def set_kernel_timing(self, enable: bool) -> None:
        _check("lopt_set_kernel_timing", load_library().lopt_set_kernel_timing(self._h, int(enable)))

    def kernel_times(self):
        """(ms[3], launches[3]) summed since the last call: row/column,
        statistics and apply kernels."""
        ms = (ctypes.c_double * 3)()
        n = (ctypes.c_int64 * 3)()
        _check("lopt_kernel_times", load_library().lopt_kernel_times(self._h, ms, n))
        return list(ms), list(n)

    def close(self) -> None:
        if getattr(self, "_h", None):
            load_library().lopt_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zeros_state(param, grad, rows: int, cols: int, weight_set: int = 0) -> TensorState:
    """State for ``param`` with zero accumulators (allocated like ``param``)."""
    import torch
    n = rows * cols
    z = lambda m: torch.zeros(m, device=param.device, dtype=torch.float32)
    return TensorState(param.reshape(-1), grad.reshape(-1), [z(n) for _ in range(3)], z(n),
                       [z(rows) for _ in range(3)], [z(cols) for _ in range(3)], rows, cols,
                       weight_set)


def rowcol_static(grad, row, col, rows: int, cols: int, inv_rho, stream=None) -> None:
    """Row/column second-moment update of one tensor through
    lopt_rowcol_static(), which allocates no device memory (its scratch is a
    fixed array inside the library).  For callers that may not call
    cudaMalloc.  ``row``/``col``: three tensors each, updated in place;
    ``inv_rho``: a 3-float tensor that receives 1 / mean(row[k])."""
    import torch
    rp = (ctypes.c_void_p * 3)(*[_ptr(r, rows, "row") for r in row])
    cp = (ctypes.c_void_p * 3)(*[_ptr(c, cols, "col") for c in col])
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check("lopt_rowcol_static", load_library().lopt_rowcol_static(
        _ptr(grad, rows * cols, "grad"), rp, cp, int(rows), int(cols), _ptr(inv_rho, 3, "inv_rho"),
        ctypes.c_void_p(handle)))
