"""Fused equivariant message passing (l <= 3) for GB300: Python binding.

A thin ctypes layer over the C ABI of ``libeqmp.so`` (declared in
include/eqmp.h).  Each function takes torch CUDA tensors, checks dtypes and
shapes, passes raw device pointers and the current CUDA stream, and raises
``EqmpError`` on a non-OK status.  All arithmetic happens in the library's
CUDA kernels; there is no CPU path.  PyTorch supplies device memory and
streams only.

Entry points (same names as the C ABI):
  eqmp_sh(vec, Y=None)                         -> Y [E, 16]
  eqmp_tp_scatter(Y, x, row_offsets, src, ...)  -> out [N, C, 16]
  eqmp_fused(vec, x, row_offsets, src, ...)     -> out [N, C, 16]
  eqmp_fused_staged(h_in, d_in, ..., out, h_out) -> h_out: copy in, layer, copy out
                                                (prepare=True: a prepared call for a step loop)
  eqmp_plan_staged(h_in, d_in, ..., out, h_out)  -> plan; plan.launch(stream): the same step as one
                                                CUDA graph launch
  eqmp_fused_so2(...)                           -> out, aligned-frame schedule
  eqmp_validate_graph(row_offsets, src, n_src, n_edges)
  eqmp_device_error()                           -> int (watchdog code)
  eqmp_fused_backward(vec, x, row_offsets, src, dst, send_offsets, send_edges, grad_out, ...)
                                                -> dict of gradients
  eqmp_fused_backward_noalloc(...)              -> the same, no workspace
  eqmp_radius_graph(pos, cutoff, box=None)      -> (dict(off, src, vec[, img, dst, rev]), E)
  eqmp_fused_lmax(l_max, vec, x, row_offsets, src, ...) -> out, degree 4..6
  eqmp_path_table()                             -> list of (l1, l2, l3)
"""
import ctypes
import os

__all__ = [
    "EqmpError", "load_library", "library_path", "eqmp_num_paths", "eqmp_path_table",
    "eqmp_status_string", "eqmp_sh", "eqmp_tp_scatter", "eqmp_fused", "eqmp_fused_staged", "eqmp_plan_staged",
    "eqmp_fused_so2",
    "eqmp_validate_graph",
    "eqmp_device_error", "eqmp_fused_backward", "eqmp_fused_backward_noalloc", "eqmp_radius_graph", "eqmp_fused_lmax",
    "eqmp_num_paths_lmax", "eqmp_watchdog_selftest", "eqmp_fp32_peak_probe", "sender_view", "EQMP_OK", "EQMP_ERR_INVALID_ARG", "EQMP_ERR_UNSUPPORTED",
    "EQMP_ERR_CUDA", "EQMP_ERR_DEVICE_TIMEOUT", "EQMP_ERR_GRAPH",
]

EQMP_OK, EQMP_ERR_INVALID_ARG, EQMP_ERR_UNSUPPORTED, EQMP_ERR_CUDA = 0, 1, 2, 3
EQMP_ERR_DEVICE_TIMEOUT, EQMP_ERR_GRAPH = 4, 5
EQMP_F32, EQMP_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
# EQMP_LIB selects another build of the library (e.g. a tuning variant).
_LIB_PATH = os.environ.get("EQMP_LIB") or os.path.join(_HERE, "_build", "libeqmp.so")
_lib = None


class EqmpError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {_status_text(status)} (status {status})")


class Weights(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("R", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("K", ctypes.c_int32)]


def library_path():
    return _LIB_PATH


def load_library():
    """Load libeqmp.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libeqmp.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.eqmp_num_paths.restype = i32
    lib.eqmp_path_table.argtypes = [ctypes.POINTER(i32)]
    lib.eqmp_path_table.restype = i32
    lib.eqmp_status_string.argtypes = [i32]
    lib.eqmp_status_string.restype = ctypes.c_char_p
    lib.eqmp_sh.argtypes = [vp, i64, vp, vp]
    lib.eqmp_sh.restype = i32
    layer = [vp, vp, i64, i32, vp, vp, i64, i64, i32, Weights, vp, i32, vp]
    lib.eqmp_tp_scatter.argtypes = layer
    lib.eqmp_tp_scatter.restype = i32
    lib.eqmp_fused.argtypes = layer
    lib.eqmp_fused.restype = i32
    lib.eqmp_fused_so2.argtypes = layer
    lib.eqmp_fused_so2.restype = i32
    sz = ctypes.c_size_t
    lib.eqmp_fused_staged.argtypes = [vp, vp, sz] + layer[:-1] + [vp, sz, vp]
    lib.eqmp_fused_staged.restype = i32
    lib.eqmp_plan_staged.argtypes = [vp, vp, sz] + layer[:-1] + [vp, sz, ctypes.POINTER(vp)]
    lib.eqmp_plan_staged.restype = i32
    lib.eqmp_plan_launch.argtypes = [vp, vp]
    lib.eqmp_plan_launch.restype = i32
    lib.eqmp_plan_destroy.argtypes = [vp]
    lib.eqmp_plan_destroy.restype = i32
    lib.eqmp_validate_graph.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.eqmp_validate_graph.restype = i32
    lib.eqmp_device_error.argtypes = [ctypes.POINTER(i32)]
    lib.eqmp_device_error.restype = i32
    lib.eqmp_fused_backward_workspace_size.argtypes = [i64, i64, i32, i32]
    lib.eqmp_fused_backward_workspace_size.restype = i64
    lib.eqmp_fused_backward.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64, i32, Weights,
                                        vp, vp, vp, vp, vp, vp, vp, i64, vp]
    lib.eqmp_fused_backward.restype = i32
    lib.eqmp_fused_backward_noalloc.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64, i32, Weights,
                                                vp, vp, vp, vp, vp, vp, vp]
    lib.eqmp_fused_backward_noalloc.restype = i32
    lib.eqmp_fused_backward_noalloc_max_bytes.restype = i64
    lib.eqmp_watchdog_selftest.argtypes = [i32, vp]
    lib.eqmp_watchdog_selftest.restype = i32
    lib.eqmp_fp32_peak_probe.argtypes = [i32, i32, vp, ctypes.POINTER(ctypes.c_double), vp]
    lib.eqmp_fp32_peak_probe.restype = i32
    lib.eqmp_num_paths_lmax.argtypes = [i32]
    lib.eqmp_num_paths_lmax.restype = i32
    lib.eqmp_fused_lmax.argtypes = [i32, vp, vp, i64, vp, vp, i64, i64, i32, Weights, vp, vp]
    lib.eqmp_fused_lmax.restype = i32
    lib.eqmp_radius_graph_workspace_size.argtypes = [i64]
    lib.eqmp_radius_graph_workspace_size.restype = ctypes.c_size_t
    lib.eqmp_radius_graph.argtypes = [vp, i64, ctypes.c_float, vp, vp, vp, vp, vp, i64, vp, vp,
                                      ctypes.c_size_t, vp]
    lib.eqmp_radius_graph.restype = i32
    lib.eqmp_radius_graph_pbc.argtypes = [vp, i64, ctypes.c_float, ctypes.POINTER(ctypes.c_float), vp, vp, vp, vp,
                                          vp, vp, i64, vp, vp, ctypes.c_size_t, vp]
    lib.eqmp_radius_graph_pbc.restype = i32
    _lib = lib
    return lib


def _status_text(status):
    try:
        return load_library().eqmp_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library absent
        return "status"


def _check(status, where):
    if status != EQMP_OK:
        raise EqmpError(status, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _require(t, name, dtype=None, cuda=True):
    import torch

    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def eqmp_num_paths():
    return int(load_library().eqmp_num_paths())


def eqmp_path_table():
    lib = load_library()
    buf = (ctypes.c_int32 * (3 * 34))()
    _check(lib.eqmp_path_table(buf), "eqmp_path_table")
    return [tuple(buf[3 * p:3 * p + 3]) for p in range(lib.eqmp_num_paths())]


def eqmp_status_string(status):
    return load_library().eqmp_status_string(int(status)).decode()


def eqmp_sh(vec, Y=None, stream=None):
    """Y[E, 16] = real SH (l <= 3) of vec[E, 3] (fp32, CUDA)."""
    import torch

    _require(vec, "vec", torch.float32)
    E = vec.shape[0] if vec.dim() == 2 else -1
    if vec.dim() != 2 or vec.shape[1] != 3:
        raise ValueError("vec must be [E, 3]")
    if Y is None:
        Y = torch.empty((E, 16), dtype=torch.float32, device=vec.device)
    _require(Y, "Y", torch.float32)
    if tuple(Y.shape) != (E, 16):
        raise ValueError("Y must be [E, 16]")
    _check(load_library().eqmp_sh(_ptr(vec), E, _ptr(Y), _stream(stream)), "eqmp_sh")
    return Y


def _layer(fn_name, edge_in, x, row_offsets, src, w, R, M, out, stream, n_edges):
    import torch

    _require(x, "x", (torch.float32, torch.bfloat16))
    _require(row_offsets, "row_offsets", torch.int32)
    _require(src, "src", torch.int32)
    for name, t in (("w", w), ("R", R), ("M", M)):
        _require(t, name, torch.float32)
    if x.dim() != 3 or x.shape[2] != 16:
        raise ValueError("x must be [N_src, C, 16]")
    n_src, C = x.shape[0], x.shape[1]
    N = row_offsets.shape[0] - 1
    E = n_edges if n_edges is not None else edge_in.shape[0]
    if out is None:
        out = torch.empty((N, C, 16), dtype=x.dtype, device=x.device)
    _require(out, "out", x.dtype)
    if tuple(out.shape) != (N, C, 16):
        raise ValueError("out must be [N, C, 16]")
    dt = EQMP_BF16 if x.dtype == torch.bfloat16 else EQMP_F32
    if w is not None:
        wt = Weights(ctypes.c_void_p(w.data_ptr()), None, None, 0)
    else:
        wt = Weights(None, ctypes.c_void_p(R.data_ptr()) if R is not None else None,
                     ctypes.c_void_p(M.data_ptr()) if M is not None else None,
                     R.shape[1] if R is not None and R.dim() == 2 else 0)
    fn = getattr(load_library(), fn_name)
    st = fn(_ptr(edge_in), _ptr(x), n_src, dt, _ptr(row_offsets), _ptr(src), N, E, C, wt,
            _ptr(out), dt, _stream(stream))
    _check(st, fn_name)
    return out


def eqmp_tp_scatter(Y, x, row_offsets, src, w=None, R=None, M=None, out=None, stream=None,
                    n_edges=None):
    """out[N, C, 16] = receiver sum of CG(x[src], Y) with shared w or radial (R, M)."""
    import torch

    _require(Y, "Y", torch.float32)
    return _layer("eqmp_tp_scatter", Y, x, row_offsets, src, w, R, M, out, stream, n_edges)


def eqmp_fused(vec, x, row_offsets, src, w=None, R=None, M=None, out=None, stream=None,
               n_edges=None):
    """out[N, C, 16] = receiver sum of CG(x[src], SH(vec)), one fused kernel."""
    import torch

    _require(vec, "vec", torch.float32)
    return _layer("eqmp_fused", vec, x, row_offsets, src, w, R, M, out, stream, n_edges)


def eqmp_fused_staged(h_in, d_in, vec, x, row_offsets, src, out, h_out, w=None, R=None, M=None, stream=None,
                      n_edges=None, prepare=False):
    """One step from host memory: h_in (pinned CPU uint8) -> d_in (CUDA
    uint8, same size), eqmp_fused on the CUDA tensors given (views into
    d_in), out -> h_out (pinned CPU, out's size).  Asynchronous on the
    stream; synchronise before reading h_out.

    prepare=True checks and marshals the arguments once and returns a
    function of no arguments that issues the same C call (for a loop that
    repeats the step on the same buffers; the tensors must stay alive and
    unmoved while it is used).  It raises EqmpError on a non-OK status."""
    import torch

    _require(h_in, "h_in", torch.uint8, cuda=False)
    _require(d_in, "d_in", torch.uint8)
    _require(h_out, "h_out", out.dtype, cuda=False)
    _require(vec, "vec", torch.float32)
    _require(x, "x", (torch.float32, torch.bfloat16))
    _require(row_offsets, "row_offsets", torch.int32)
    _require(src, "src", torch.int32)
    for name, t in (("w", w), ("R", R), ("M", M)):
        _require(t, name, torch.float32)
    if h_in.is_cuda or h_out.is_cuda:
        raise ValueError("h_in and h_out are host tensors")
    if h_in.numel() != d_in.numel():
        raise ValueError("h_in and d_in must have the same size")
    if x.dim() != 3 or x.shape[2] != 16:
        raise ValueError("x must be [N_src, C, 16]")
    n_src, C = x.shape[0], x.shape[1]
    N = row_offsets.shape[0] - 1
    E = n_edges if n_edges is not None else vec.shape[0]
    _require(out, "out", x.dtype)
    if tuple(out.shape) != (N, C, 16) or tuple(h_out.shape) != (N, C, 16):
        raise ValueError("out and h_out must be [N, C, 16]")
    dt = EQMP_BF16 if x.dtype == torch.bfloat16 else EQMP_F32
    if w is not None:
        wt = Weights(ctypes.c_void_p(w.data_ptr()), None, None, 0)
    else:
        wt = Weights(None, ctypes.c_void_p(R.data_ptr()) if R is not None else None,
                     ctypes.c_void_p(M.data_ptr()) if M is not None else None,
                     R.shape[1] if R is not None and R.dim() == 2 else 0)
    fn = load_library().eqmp_fused_staged
    args = (_ptr(h_in), _ptr(d_in), h_in.numel(), _ptr(vec), _ptr(x), n_src, dt, _ptr(row_offsets), _ptr(src),
            N, E, C, wt, _ptr(out), dt, _ptr(h_out), h_out.numel() * h_out.element_size(), _stream(stream))
    if prepare == "plan":
        return _Plan(args[:-1], (h_in, d_in, vec, x, row_offsets, src, out, h_out, w, R, M))
    if prepare:
        keep = (h_in, d_in, vec, x, row_offsets, src, out, h_out, w, R, M, stream)

        def run(_keep=keep):
            st = fn(*args)
            if st != EQMP_OK:
                raise EqmpError(st, "eqmp_fused_staged")
            return h_out
        return run
    _check(fn(*args), "eqmp_fused_staged")
    return h_out


class _Plan:
    """A staged step recorded once as a CUDA graph (eqmp_plan_staged);
    launch(stream) replays it with one graph launch."""

    def __init__(self, args, keep):
        lib = load_library()
        h = ctypes.c_void_p()
        _check(lib.eqmp_plan_staged(*args, ctypes.byref(h)), "eqmp_plan_staged")
        self._h, self._keep, self._lib = h, keep, lib
        self.h_out = keep[7]

    def launch(self, stream=None):
        st = self._lib.eqmp_plan_launch(self._h, _stream(stream))
        if st != EQMP_OK:
            raise EqmpError(st, "eqmp_plan_launch")
        return self.h_out

    def destroy(self):
        if self._h:
            self._lib.eqmp_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def eqmp_plan_staged(h_in, d_in, vec, x, row_offsets, src, out, h_out, w=None, R=None, M=None, n_edges=None):
    """The step of eqmp_fused_staged recorded once as a CUDA graph: returns a
    plan whose launch(stream=None) replays the input copy, the layer and the
    result copy with one graph launch.  The tensors must stay alive and
    unmoved while the plan is used (the plan holds references to them);
    h_in and h_out must be pinned."""
    if not (h_in.is_pinned() and h_out.is_pinned()):
        raise ValueError("h_in and h_out must be pinned for a plan")
    return eqmp_fused_staged(h_in, d_in, vec, x, row_offsets, src, out, h_out, w=w, R=R, M=M, n_edges=n_edges,
                             prepare="plan")


def eqmp_fused_so2(vec, x, row_offsets, src, w=None, R=None, M=None, out=None, stream=None,
                   n_edges=None):
    """eqmp_fused computed in the aligned (SO(2)) edge frame; same result."""
    import torch

    _require(vec, "vec", torch.float32)
    return _layer("eqmp_fused_so2", vec, x, row_offsets, src, w, R, M, out, stream, n_edges)


def eqmp_validate_graph(row_offsets, src, n_src, n_edges, stream=None):
    """Raise EqmpError(EQMP_ERR_GRAPH) if the CSR preconditions do not hold."""
    N = row_offsets.shape[0] - 1
    st = load_library().eqmp_validate_graph(_ptr(row_offsets), _ptr(src), N, int(n_src),
                                            int(n_edges), _stream(stream))
    _check(st, "eqmp_validate_graph")


def eqmp_device_error():
    """Watchdog code since the last call (0 = no device wait gave up)."""
    code = ctypes.c_int32(0)
    st = load_library().eqmp_device_error(ctypes.byref(code))
    if st not in (EQMP_OK, EQMP_ERR_DEVICE_TIMEOUT):
        _check(st, "eqmp_device_error")
    return int(code.value)


def eqmp_watchdog_selftest(wait_ms=20, stream=None):
    """Launch the watchdog self-test (a wait that must give up); read the code with eqmp_device_error()."""
    _check(load_library().eqmp_watchdog_selftest(int(wait_ms), _stream(stream)), "eqmp_watchdog_selftest")


def eqmp_fp32_peak_probe(iters, out, blocks_per_sm=4, stream=None):
    """Launch the FP32 throughput probe (out: one-float CUDA tensor); returns its flop count."""
    flops = ctypes.c_double(0.0)
    _check(load_library().eqmp_fp32_peak_probe(int(iters), int(blocks_per_sm), _ptr(out), ctypes.byref(flops),
                                                _stream(stream)), "eqmp_fp32_peak_probe")
    return flops.value


def eqmp_num_paths_lmax(l_max):
    return int(load_library().eqmp_num_paths_lmax(int(l_max)))


def eqmp_fused_lmax(l_max, vec, x, row_offsets, src, w=None, R=None, M=None, out=None, stream=None):
    """The layer at degree l_max = 4..6: x [N_src, C, (l_max+1)^2] fp32 -> out [N, C, (l_max+1)^2]."""
    import torch

    l_max = int(l_max)
    nc = (l_max + 1) ** 2
    for name, t in (("vec", vec), ("x", x), ("w", w), ("R", R), ("M", M)):
        _require(t, name, torch.float32)
    _require(row_offsets, "row_offsets", torch.int32)
    _require(src, "src", torch.int32)
    if x.dim() != 3 or x.shape[2] != nc:
        raise ValueError(f"x must be [N_src, C, {nc}]")
    n_src, C = x.shape[0], x.shape[1]
    N = row_offsets.shape[0] - 1
    if out is None:
        out = torch.empty((N, C, nc), dtype=torch.float32, device=x.device)
    _require(out, "out", torch.float32)
    if tuple(out.shape) != (N, C, nc):
        raise ValueError(f"out must be [N, C, {nc}]")
    if w is not None:
        wt = Weights(ctypes.c_void_p(w.data_ptr()), None, None, 0)
    else:
        wt = Weights(None, ctypes.c_void_p(R.data_ptr()) if R is not None else None,
                     ctypes.c_void_p(M.data_ptr()) if M is not None else None,
                     R.shape[1] if R is not None and R.dim() == 2 else 0)
    st = load_library().eqmp_fused_lmax(l_max, _ptr(vec), _ptr(x), n_src, _ptr(row_offsets), _ptr(src), N,
                                        vec.shape[0], C, wt, _ptr(out), _stream(stream))
    _check(st, "eqmp_fused_lmax")
    return out


def eqmp_radius_graph(pos, cutoff, e_cap=None, dst=False, rev=False, stream=None, box=None):
    """Radius graph of pos [N, 3] fp32 (CUDA): dict(off, src, vec[, img][, dst][, rev]), E.

    Edges j -> i for i != j with the float32 squared distance below
    cutoff^2, CSR by receiver with senders ascending.  With box = (Lx, Ly, Lz)
    the boundaries are periodic (eqmp_radius_graph_pbc): positions inside the
    box, every image within one box length per direction, and "img" holds
    each edge's image index.  When the edge count exceeds the capacity
    (e_cap, default 64 N), the call is repeated once with the exact count,
    which costs one device-to-host read of E.
    """
    import torch

    _require(pos, "pos", torch.float32)
    if pos.dim() != 2 or pos.shape[1] != 3:
        raise ValueError("pos must be [N, 3]")
    lib = load_library()
    N = pos.shape[0]
    dev = pos.device
    ws = torch.empty(max(int(lib.eqmp_radius_graph_workspace_size(N)), 256), dtype=torch.uint8, device=dev)
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    e_total = torch.empty(1, dtype=torch.int64, device=dev)
    cap = int(64 * N if e_cap is None else e_cap)
    st = _stream(stream)
    for _ in range(2):
        out = dict(off=off, src=torch.empty(cap, dtype=torch.int32, device=dev),
                   vec=torch.empty((cap, 3), dtype=torch.float32, device=dev))
        if dst:
            out["dst"] = torch.empty(cap, dtype=torch.int32, device=dev)
        if rev:
            out["rev"] = torch.empty(cap, dtype=torch.int32, device=dev)
        if box is None:
            _check(lib.eqmp_radius_graph(_ptr(pos), N, float(cutoff), _ptr(off), _ptr(out["src"]),
                                         _ptr(out["vec"]), _ptr(out.get("dst")), _ptr(out.get("rev")), cap,
                                         _ptr(e_total), _ptr(ws), ws.numel(), st), "eqmp_radius_graph")
        else:
            out["img"] = torch.empty(cap, dtype=torch.int32, device=dev)
            lengths = (ctypes.c_float * 3)(*[float(v) for v in box])
            _check(lib.eqmp_radius_graph_pbc(_ptr(pos), N, float(cutoff), lengths, _ptr(off), _ptr(out["src"]),
                                             _ptr(out["vec"]), _ptr(out["img"]), _ptr(out.get("dst")),
                                             _ptr(out.get("rev")), cap, _ptr(e_total), _ptr(ws), ws.numel(), st),
                   "eqmp_radius_graph_pbc")
        E = int(e_total.item())
        if E < 0:
            raise EqmpError(EQMP_ERR_INVALID_ARG, "eqmp_radius_graph: positions non-finite or out of range"
                            " (outside the box, with periodic boundaries)"
                            if E == -1 else "eqmp_radius_graph: 2^31 edges or more")
        if E <= cap:
            break
        cap = E
    for k in ("src", "vec", "img", "dst", "rev"):
        if k in out:
            out[k] = out[k][:E]
    return out, E


def sender_view(src, n_src):
    """(send_offsets [n_src+1], send_edges [E]) grouping edge ids by sender
    (stable, edge order kept within a sender); host-side graph preparation
    for eqmp_fused_backward (numpy or torch CPU int arrays in, numpy out)."""
    import numpy as np

    src = np.asarray(src, dtype=np.int64)
    order = np.argsort(src, kind="stable").astype(np.int32)
    offs = np.searchsorted(src[order], np.arange(int(n_src) + 1), side="left").astype(np.int32)
    return offs, order


def _backward_prepare(vec, x, row_offsets, src, dst, send_offsets, send_edges, grad_out, w, R, M, need):
    """Checks of the backward's inputs and its requested output tensors."""
    import torch

    spec = (("vec", vec, torch.float32), ("x", x, torch.float32),
            ("row_offsets", row_offsets, torch.int32), ("src", src, torch.int32),
            ("dst", dst, torch.int32), ("send_offsets", send_offsets, torch.int32),
            ("send_edges", send_edges, torch.int32), ("grad_out", grad_out, torch.float32),
            ("w", w, torch.float32), ("R", R, torch.float32), ("M", M, torch.float32))
    for name, t, dt in spec:  # every dtype first, then placement and layout
        _require(t, name, dt, cuda=False)
    for name, t, dt in spec:
        _require(t, name, dt)
    if (w is None) == (R is None or M is None):
        raise ValueError("give exactly one of w or (R, M)")
    n_src, C = x.shape[0], x.shape[1]
    N = row_offsets.shape[0] - 1
    E = vec.shape[0]
    radial = w is None
    dev = x.device
    out = {}
    if "x" in need:
        out["x"] = torch.empty((n_src, C, 16), dtype=torch.float32, device=dev)
    if "vec" in need:
        out["vec"] = torch.zeros((E, 3), dtype=torch.float32, device=dev)
    if radial:
        if "R" in need:
            out["R"] = torch.zeros((E, 8), dtype=torch.float32, device=dev)
        if "M" in need:
            out["M"] = torch.empty((8, 34 * C), dtype=torch.float32, device=dev)
    elif "w" in need:
        out["w"] = torch.empty((34, C), dtype=torch.float32, device=dev)
    wt = (Weights(ctypes.c_void_p(w.data_ptr()), None, None, 0) if not radial else
          Weights(None, ctypes.c_void_p(R.data_ptr()), ctypes.c_void_p(M.data_ptr()), R.shape[1]))
    head = (_ptr(vec), _ptr(x), n_src, _ptr(row_offsets), _ptr(src), _ptr(dst), _ptr(send_offsets),
            _ptr(send_edges), send_edges.shape[0], N, E, C, wt, _ptr(grad_out), _ptr(out.get("x")),
            _ptr(out.get("w")), _ptr(out.get("R")), _ptr(out.get("M")), _ptr(out.get("vec")))
    return out, head, (N, E, C, radial)


def eqmp_fused_backward(vec, x, row_offsets, src, dst, send_offsets, send_edges, grad_out,
                        w=None, R=None, M=None, need=("x", "w", "vec"), stream=None):
    """Gradients of the fused layer; returns {"x", "w" | "R", "M", "vec"} as requested."""
    import torch

    out, head, (N, E, C, radial) = _backward_prepare(vec, x, row_offsets, src, dst, send_offsets,
                                                     send_edges, grad_out, w, R, M, need)
    lib = load_library()
    nbytes = int(lib.eqmp_fused_backward_workspace_size(N, E, C, 1 if radial else 0))
    if nbytes < 0:
        raise EqmpError(EQMP_ERR_CUDA, "eqmp_fused_backward_workspace_size")
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=x.device)
    _check(lib.eqmp_fused_backward(*head, _ptr(ws), ws.numel() * 4, _stream(stream)), "eqmp_fused_backward")
    return out


def eqmp_fused_backward_noalloc(vec, x, row_offsets, src, dst, send_offsets, send_edges, grad_out,
                                w=None, R=None, M=None, need=("x", "w", "vec"), stream=None):
    """eqmp_fused_backward with the library's static scratch instead of a
    workspace (the C entry point allocates no device memory; this wrapper
    only allocates the requested output tensors through torch)."""
    out, head, _ = _backward_prepare(vec, x, row_offsets, src, dst, send_offsets, send_edges, grad_out,
                                     w, R, M, need)
    _check(load_library().eqmp_fused_backward_noalloc(*head, _stream(stream)), "eqmp_fused_backward_noalloc")
    return out
