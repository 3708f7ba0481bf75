"""Blockwise-FP8 linear layer for B300 (sm_103a): Python binding of the C ABI in include/bfp8.h.

The binding only marshals arguments: it takes CUDA tensors (torch is used for
device memory and streams), allocates outputs when none are given, and calls
``libbfp8.so`` through ctypes on the current torch stream. Every step of the
path runs in the library's CUDA kernels; there is no CPU fallback. If the
library is missing or the device is not a B300, calls raise.

Entry points (same names as the C ABI):
  fp8_quantize_act(x)            -> (q [R,C] u8, s [C/128, R] f32)
  fp8_quantize_weight(w)         -> (q [N,K] u8, s [N/128, K/128] f32)
  fp8_quantize_transpose(x)      -> (qt [C, R128] u8, st [R128/128, C] f32)
  fp8_quantize_act_transpose(x)  -> (q, s, qt, st): both layouts, one read of x
  fp8_block_gemm_fwd(qx, sx, qw, sw)        -> y  [M, N] bf16
  fp8_block_gemm_dgrad(qdy, sdy, qw, sw)    -> dx [M, K] bf16
  fp8_block_gemm_wgrad(qdyt, sdyt, qxt, sxt, M) -> dw [N, K] bf16
    (each takes an optional workspace=gemm_workspace(): the split of the grid's
    last partial round of tiles along the contraction axis)
  fp8_block_gemm_wgrad_acc(qdyt, sdyt, qxt, sxt, M, main_grad): main_grad [N, K] f32 += dW
MuonH (one optimizer step for one weight matrix):
  muonh_update(w, g, lr, radius)  # w FP32 in place; see muonh_update's docstring
  bf16_gemm_axpby(a, b, c, alpha, beta) -> d = alpha a b + beta c (BF16, FP32 sums)
  muonh_newton_schulz(x)          # Newton-Schulz iterations on a BF16 matrix, in place
Scale tensors are allocated with a row stride rounded up to 4 elements so that
the GEMMs' TMA loads see 16-byte rows; the returned tensors are views of the
valid columns.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
LIB_PATH = os.path.join(_PKG, "libbfp8.so")
HEADER_PATH = os.path.join(_ROOT, "include", "bfp8.h")
TILE = 128

STATUS = {0: "BFP8_OK", -1: "BFP8_EINVAL", -2: "BFP8_EALIGN", -3: "BFP8_ESHAPE",
          -4: "BFP8_ELAUNCH", -5: "BFP8_ETIMEOUT", -6: "BFP8_EARCH"}


class Bfp8Error(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libbfp8.so and declare its signatures. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libbfp8.so not found at {path}; build it with "
                          f"`python -m blockwise_fp8_linear_weight_b300.build`")
    lib = ctypes.CDLL(path)
    i64, p, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sig = {
        "fp8_quantize_act": [p, i64, i64, i64, p, i64, p, i64, p],
        "fp8_quantize_weight": [p, i64, i64, i64, p, i64, p, p],
        "fp8_quantize_transpose": [p, i64, i64, i64, p, i64, p, i64, p],
        "fp8_quantize_act_transpose": [p, i64, i64, i64, p, i64, p, i64, p, i64, p, i64, p],
        "fp8_block_gemm_workspace_bytes": [ctypes.POINTER(i64)],
        "fp8_block_gemm_fwd": [p, i64, p, i64, p, i64, p, p, i64, i64, i64, i64, p, i64, p],
        "fp8_block_gemm_dgrad": [p, i64, p, i64, p, i64, p, p, i64, i64, i64, i64, p, i64, p],
        "fp8_block_gemm_wgrad": [p, i64, p, i64, p, i64, p, i64, p, i64, i64, i64, i64, p, i64, p],
        "fp8_block_gemm_wgrad_acc": [p, i64, p, i64, p, i64, p, i64, p, i64, i64, i64, i64, p],
        "bfp8_last_device_status": [p],
        "bfp8_set_gemm_tile_n": [c_int],
        "bfp8_set_wait_limit_ns": [i64],
        "bfp8_test_stall_producers": [c_int],
        "bfp8_kernel_launches": [ctypes.POINTER(i64)],
        "muonh_partials_len": [ctypes.POINTER(c_int)],
        "muonh_normalize": [p, i64, i64, i64, p, i64, p, i64, ctypes.c_float, p],
        "muonh_apply": [p, i64, p, i64, i64, i64, p, i64, ctypes.c_float, ctypes.c_float, p],
        "muonh_apply_static": [p, i64, p, i64, i64, i64, ctypes.c_float, ctypes.c_float, p],
        "bf16_gemm_axpby": [p, i64, p, i64, c_int, p, i64, p, i64, i64, i64, i64, ctypes.c_float, ctypes.c_float, p],
        "muonh_newton_schulz_work_bytes": [i64, i64, ctypes.POINTER(i64)],
        "muonh_newton_schulz": [p, i64, i64, i64, p, i64, c_int, ctypes.c_float, ctypes.c_float, ctypes.c_float, p],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = c_int
    lib.bfp8_status_string.argtypes = [c_int]
    lib.bfp8_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def header_functions(path: str = HEADER_PATH):
    """Names of the functions declared in include/bfp8.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def _check(fn: str, rc: int):
    if rc != 0:
        msg = load_library().bfp8_status_string(rc).decode()
        raise Bfp8Error(fn, rc, msg)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _req(t, dtype, name, ndim=2):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or (ndim == 2 and t.stride(1) != 1):
        raise ValueError(f"{name} must be a row-major 2-D tensor with unit column stride")
    return t


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def _scales(chunks: int, n: int, device):
    """[chunks, n] float32 view of a buffer whose row stride is n rounded up to 4."""
    buf = torch.empty((chunks, max(_round_up(n, 4), 4)), dtype=torch.float32, device=device)
    return buf[:, :n]


# ----------------------------------------------------------------------- quantisers
def fp8_quantize_act(x, q=None, s=None):
    """1x128 tiles along the columns of x [R, C] (bf16). Returns (q, s)."""
    lib = load_library()
    _req(x, torch.bfloat16, "x")
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device) if q is None else q
    s = _scales(C // TILE if C % TILE == 0 else 0, R, x.device) if s is None else s
    _check("fp8_quantize_act", lib.fp8_quantize_act(
        _ptr(x), R, C, x.stride(0), _ptr(q), q.stride(0), _ptr(s), s.stride(0), _stream()))
    return q, s


def fp8_quantize_weight(w, q=None, s=None):
    """128x128 blocks of w [N, K] (bf16). Returns (q, s) with s [N/128, K/128]."""
    lib = load_library()
    _req(w, torch.bfloat16, "w")
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty((N // TILE, K // TILE), dtype=torch.float32, device=w.device) if s is None else s
    if s.dim() != 2 or not s.is_contiguous():
        raise ValueError("weight scales must be a dense [N/128, K/128] tensor")
    _check("fp8_quantize_weight", lib.fp8_quantize_weight(
        _ptr(w), N, K, w.stride(0), _ptr(q), q.stride(0), _ptr(s), _stream()))
    return q, s


def fp8_quantize_transpose(x, qt=None, st=None):
    """Tiles of 128 rows of x [R, C] (bf16), written transposed. Returns (qt [C, R128], st [R128/128, C])."""
    lib = load_library()
    _req(x, torch.bfloat16, "x")
    R, C = x.shape
    R128 = _round_up(R, TILE)
    qt = torch.empty((C, R128), dtype=torch.uint8, device=x.device) if qt is None else qt
    if st is None:
        st = torch.empty((R128 // TILE, _round_up(C, 4)), dtype=torch.float32, device=x.device)[:, :C]
    _check("fp8_quantize_transpose", lib.fp8_quantize_transpose(
        _ptr(x), R, C, x.stride(0), _ptr(qt), qt.stride(0), _ptr(st), st.stride(0), _stream()))
    return qt, st


def fp8_quantize_act_transpose(x, q=None, s=None, qt=None, st=None):
    """Both layouts of x [R, C] (bf16) in one pass: (q, s) as fp8_quantize_act, (qt, st) as
    fp8_quantize_transpose."""
    lib = load_library()
    _req(x, torch.bfloat16, "x")
    R, C = x.shape
    R128 = _round_up(R, TILE)
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device) if q is None else q
    s = _scales(C // TILE if C % TILE == 0 else 0, R, x.device) if s is None else s
    qt = torch.empty((C, R128), dtype=torch.uint8, device=x.device) if qt is None else qt
    if st is None:
        st = torch.empty((R128 // TILE, _round_up(C, 4)), dtype=torch.float32, device=x.device)[:, :C]
    _check("fp8_quantize_act_transpose", lib.fp8_quantize_act_transpose(
        _ptr(x), R, C, x.stride(0), _ptr(q), q.stride(0), _ptr(s), s.stride(0),
        _ptr(qt), qt.stride(0), _ptr(st), st.stride(0), _stream()))
    return q, s, qt, st


# ----------------------------------------------------------------------- GEMMs
def gemm_workspace_bytes() -> int:
    """Workspace size that lets the GEMMs split their last partial round of tiles (current device)."""
    n = ctypes.c_int64(0)
    _check("fp8_block_gemm_workspace_bytes", load_library().fp8_block_gemm_workspace_bytes(ctypes.byref(n)))
    return n.value


def gemm_workspace(device="cuda"):
    """A GEMM workspace (uint8 CUDA tensor) for the device; calls sharing one must be stream-ordered."""
    with torch.cuda.device(torch.device(device)):
        return torch.empty(gemm_workspace_bytes(), dtype=torch.uint8, device=device)


def _ws(workspace):
    if workspace is None:
        return None, 0
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def fp8_block_gemm_fwd(qx, sx, qw, sw, y=None, workspace=None):
    """y [M, N] bf16 = blockwise-FP8 x W^T from (qx [M,K], sx [K/128, M], qw [N,K], sw [N/128, K/128])."""
    lib = load_library()
    M, K = qx.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device) if y is None else y
    ws, ws_bytes = _ws(workspace)
    _check("fp8_block_gemm_fwd", lib.fp8_block_gemm_fwd(
        _ptr(qx), qx.stride(0), _ptr(sx), sx.stride(0), _ptr(qw), qw.stride(0), _ptr(sw),
        _ptr(y), y.stride(0), M, N, K, ws, ws_bytes, _stream()))
    return y


def fp8_block_gemm_dgrad(qdy, sdy, qw, sw, dx=None, workspace=None):
    """dx [M, K] bf16 = blockwise-FP8 dy W from (qdy [M,N], sdy [N/128, M], qw [N,K], sw [N/128, K/128])."""
    lib = load_library()
    M, N = qdy.shape
    K = qw.shape[1]
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=qdy.device) if dx is None else dx
    ws, ws_bytes = _ws(workspace)
    _check("fp8_block_gemm_dgrad", lib.fp8_block_gemm_dgrad(
        _ptr(qdy), qdy.stride(0), _ptr(sdy), sdy.stride(0), _ptr(qw), qw.stride(0), _ptr(sw),
        _ptr(dx), dx.stride(0), M, N, K, ws, ws_bytes, _stream()))
    return dx


def fp8_block_gemm_wgrad(qdyt, sdyt, qxt, sxt, M, dw=None, workspace=None):
    """dw [N, K] bf16 = blockwise-FP8 dy^T x from transposed tiles (qdyt [N,M128], qxt [K,M128])."""
    lib = load_library()
    N = qdyt.shape[0]
    K = qxt.shape[0]
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=qdyt.device) if dw is None else dw
    ws, ws_bytes = _ws(workspace)
    _check("fp8_block_gemm_wgrad", lib.fp8_block_gemm_wgrad(
        _ptr(qdyt), qdyt.stride(0), _ptr(sdyt), sdyt.stride(0), _ptr(qxt), qxt.stride(0),
        _ptr(sxt), sxt.stride(0), _ptr(dw), dw.stride(0), M, N, K, ws, ws_bytes, _stream()))
    return dw


def fp8_block_gemm_wgrad_acc(qdyt, sdyt, qxt, sxt, M, main_grad):
    """main_grad [N, K] f32 += blockwise-FP8 dy^T x (FP32 sum, no BF16 rounding), in place."""
    lib = load_library()
    N = qdyt.shape[0]
    K = qxt.shape[0]
    _req(main_grad, torch.float32, "main_grad")
    _check("fp8_block_gemm_wgrad_acc", lib.fp8_block_gemm_wgrad_acc(
        _ptr(qdyt), qdyt.stride(0), _ptr(sdyt), sdyt.stride(0), _ptr(qxt), qxt.stride(0),
        _ptr(sxt), sxt.stride(0), _ptr(main_grad), main_grad.stride(0), M, N, K, _stream()))
    return main_grad


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far (host-side count)."""
    n = ctypes.c_int64(0)
    _check("bfp8_kernel_launches", load_library().bfp8_kernel_launches(ctypes.byref(n)))
    return n.value


def last_device_status() -> int:
    """Synchronise the current stream and read/clear the kernels' bounded-wait status word."""
    return load_library().bfp8_last_device_status(_stream())


def set_wait_limit_ns(ns: int) -> None:
    """Limit of one in-kernel pipeline wait in ns (0 = the default 2 s)."""
    _check("bfp8_set_wait_limit_ns", load_library().bfp8_set_wait_limit_ns(int(ns)))


def test_stall_producers(on: bool) -> bool:
    """Test switch: later quantiser and GEMM launches load nothing, so their waits run out.
    Returns the previous setting."""
    rc = load_library().bfp8_test_stall_producers(1 if on else 0)
    if rc < 0:
        raise ValueError("on must be a bool")
    return bool(rc)


def set_gemm_tile_n(tile_n: int) -> int:
    """GEMM output tile width: 0 (automatic), 128, 192 or 256. Returns the previous value."""
    rc = load_library().bfp8_set_gemm_tile_n(int(tile_n))
    if rc < 0:
        raise ValueError("tile_n must be 0, 128, 192 or 256")
    return rc


# ----------------------------------------------------------------------- one linear layer
class BlockwiseFP8Linear:
    """Buffers and call sequence of one blockwise-FP8 linear layer y = x W^T (x [M,K], W [N,K]).

    ``forward(x, w)`` quantises x in both layouts (1x128 along K for the
    forward GEMM, 1x128 along M, transposed, for the weight-gradient GEMM) and
    W (128x128), then runs the forward GEMM; ``backward(dy)`` quantises dy in
    both layouts and runs the input- and weight-gradient GEMMs. All outputs
    live in buffers allocated once, so a training step launches six kernels
    (plus one tail-reduce kernel per GEMM whose last round of tiles is split)
    and allocates nothing.

    Options:
      reuse_weight_quant: keep W's codes and scales while W is unchanged (same
        storage, same torch version counter), so that micro-batches after the
        first of an optimizer step skip the weight quantiser (five kernels).
        The FP8 copy is derived, non-persistent state: it is rebuilt from W
        whenever W changes and never needs saving.
      main_grad: accumulate dW into an FP32 main-gradient buffer
        (``self.main_grad``, zeroed by ``zero_main_grad()``) instead of writing
        a BF16 dW, as a trainer keeping its state in FP32 does across
        micro-batches.
      workspace: the GEMM workspace (``gemm_workspace()``, 38 MB on a B300)
        that lets each GEMM split the grid's last partial round of tiles along
        the contraction axis; layers that run one after another on one stream
        may share one. None: allocate one for this layer. False: no split.
    """

    def __init__(self, M: int, K: int, N: int, device="cuda", reuse_weight_quant: bool = False,
                 main_grad: bool = False, workspace=None):
        self.M, self.K, self.N = M, K, N
        self.reuse_weight_quant = reuse_weight_quant
        self.weight_quant_calls = 0
        self._w_key = None
        dev = torch.device(device)
        M128 = _round_up(M, TILE)
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        self.qx = torch.empty((M, K), dtype=u8, device=dev)
        self.sx = _scales(K // TILE, M, dev)
        self.qw = torch.empty((N, K), dtype=u8, device=dev)
        self.sw = torch.empty((N // TILE, K // TILE), dtype=f32, device=dev)
        self.qdy = torch.empty((M, N), dtype=u8, device=dev)
        self.sdy = _scales(N // TILE, M, dev)
        self.qdyt = torch.empty((N, M128), dtype=u8, device=dev)
        self.sdyt = _scales(M128 // TILE, N, dev)
        self.qxt = torch.empty((K, M128), dtype=u8, device=dev)
        self.sxt = _scales(M128 // TILE, K, dev)
        self.y = torch.empty((M, N), dtype=bf, device=dev)
        self.dx = torch.empty((M, K), dtype=bf, device=dev)
        self.dw = None if main_grad else torch.empty((N, K), dtype=bf, device=dev)
        self.main_grad = torch.zeros((N, K), dtype=f32, device=dev) if main_grad else None
        if workspace is None:
            workspace = gemm_workspace(dev)
        self.workspace = workspace if workspace is not False else None

    def quantize_weight(self, w):
        """Quantise W unless reuse is on and W is the tensor (and version) quantised last."""
        key = (w.data_ptr(), w._version, tuple(w.shape), tuple(w.stride()))
        if self.reuse_weight_quant and key == self._w_key:
            return
        fp8_quantize_weight(w, self.qw, self.sw)
        self.weight_quant_calls += 1
        self._w_key = key

    def invalidate_weight_quant(self):
        """Forget the cached weight codes (e.g. after W was changed behind torch's back)."""
        self._w_key = None

    def zero_main_grad(self):
        self.main_grad.zero_()

    def forward(self, x, w):
        fp8_quantize_act_transpose(x, self.qx, self.sx, self.qxt, self.sxt)
        self.quantize_weight(w)
        fp8_block_gemm_fwd(self.qx, self.sx, self.qw, self.sw, self.y, workspace=self.workspace)
        return self.y

    def backward(self, dy):
        """Returns (dx, dW): dW is the BF16 buffer, or the FP32 main gradient it was added into."""
        fp8_quantize_act_transpose(dy, self.qdy, self.sdy, self.qdyt, self.sdyt)
        fp8_block_gemm_dgrad(self.qdy, self.sdy, self.qw, self.sw, self.dx, workspace=self.workspace)
        if self.main_grad is not None:
            fp8_block_gemm_wgrad_acc(self.qdyt, self.sdyt, self.qxt, self.sxt, self.M, self.main_grad)
            return self.dx, self.main_grad
        fp8_block_gemm_wgrad(self.qdyt, self.sdyt, self.qxt, self.sxt, self.M, self.dw,
                             workspace=self.workspace)
        return self.dx, self.dw


# ----------------------------------------------------------------------- MuonH
# Quintic Newton-Schulz coefficients of the public Muon optimizer (K. Jordan et
# al., "Muon: an optimizer for hidden layers in neural networks", 2024); the
# Puro-2B pages name MuonH but give no coefficients.
MUON_NS_COEFFS = (3.4445, -4.7750, 2.0315)


def _muonh_partials(device):
    n = ctypes.c_int(0)
    _check("muonh_partials_len", load_library().muonh_partials_len(ctypes.byref(n)))
    return torch.empty(n.value, dtype=torch.float64, device=device)


def muonh_normalize(g, x=None, eps: float = 1e-7, partials=None):
    """x = bf16(g / (|g|_F + eps)) for an FP32 matrix g [rows, cols] (cols % 4 == 0)."""
    lib = load_library()
    _req(g, torch.float32, "g")
    rows, cols = g.shape
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device=g.device) if x is None else x
    partials = _muonh_partials(g.device) if partials is None else partials
    _req(partials, torch.float64, "partials", ndim=1)
    _check("muonh_normalize", lib.muonh_normalize(_ptr(g), rows, cols, g.stride(0), _ptr(x), x.stride(0),
                                                  _ptr(partials), partials.numel(), float(eps), _stream()))
    return x


def muonh_apply(w, u, lr: float, radius: float, partials=None):
    """w = R (w - a u) / |w - a u|_F in place, a = lr R / |u|_F; w FP32, u BF16, same shape."""
    lib = load_library()
    _req(w, torch.float32, "w")
    _req(u, torch.bfloat16, "u")
    if u.shape != w.shape:
        raise ValueError("u must have w's shape")
    rows, cols = w.shape
    partials = _muonh_partials(w.device) if partials is None else partials
    _req(partials, torch.float64, "partials", ndim=1)
    _check("muonh_apply", lib.muonh_apply(_ptr(w), w.stride(0), _ptr(u), u.stride(0), rows, cols,
                                          _ptr(partials), partials.numel(), float(lr), float(radius), _stream()))
    return w


def muonh_apply_static(w, u, lr: float, radius: float):
    """muonh_apply with the library's own device scratch (calls on a device must be ordered)."""
    lib = load_library()
    _req(w, torch.float32, "w")
    _req(u, torch.bfloat16, "u")
    if u.shape != w.shape:
        raise ValueError("u must have w's shape")
    rows, cols = w.shape
    _check("muonh_apply_static", lib.muonh_apply_static(_ptr(w), w.stride(0), _ptr(u), u.stride(0), rows, cols,
                                                        float(lr), float(radius), _stream()))
    return w


def bf16_gemm_axpby(a, b, c=None, alpha: float = 1.0, beta: float = 0.0, b_mn_major: bool = False, d=None):
    """d = bf16(alpha * a @ B + beta * c) with a [M, K] and B = b^T (b [N, K]) or B = b (b [K, N],
    b_mn_major=True), all BF16; the products are summed in FP32 by the library's tcgen05 kernel."""
    lib = load_library()
    _req(a, torch.bfloat16, "a")
    _req(b, torch.bfloat16, "b")
    M, K = a.shape
    N = b.shape[1] if b_mn_major else b.shape[0]
    d = torch.empty((M, N), dtype=torch.bfloat16, device=a.device) if d is None else d
    if c is not None:
        _req(c, torch.bfloat16, "c")
    _check("bf16_gemm_axpby", lib.bf16_gemm_axpby(
        _ptr(a), a.stride(0), _ptr(b), b.stride(0), 1 if b_mn_major else 0,
        _ptr(c) if c is not None else None, c.stride(0) if c is not None else 0,
        _ptr(d), d.stride(0), M, N, K, float(alpha), float(beta), _stream()))
    return d


def muonh_newton_schulz(x, steps: int = 5, coeffs=MUON_NS_COEFFS, work=None):
    """Quintic Newton-Schulz iterations X <- a X + (b A + c A^2) X, A = X X^T, on the orientation
    with fewer rows, in place on a BF16 matrix x (rows, cols multiples of 8). Every product runs in
    the library's BF16 tcgen05 GEMM; work is a caller buffer of muonh_newton_schulz_work_bytes."""
    lib = load_library()
    _req(x, torch.bfloat16, "x")
    rows, cols = x.shape
    if work is None:
        n = ctypes.c_int64(0)
        _check("muonh_newton_schulz_work_bytes", lib.muonh_newton_schulz_work_bytes(rows, cols, ctypes.byref(n)))
        work = torch.empty(n.value, dtype=torch.uint8, device=x.device)
    a, b, c = coeffs
    _check("muonh_newton_schulz", lib.muonh_newton_schulz(
        _ptr(x), rows, cols, x.stride(0), _ptr(work), work.numel(), int(steps), float(a), float(b), float(c),
        _stream()))
    return x


def muonh_update(w, g, lr: float, radius: float, steps: int = 5, coeffs=MUON_NS_COEFFS, eps: float = 1e-7):
    """One MuonH step for one weight matrix, in place: w (FP32 [N, K]) moves by a relative
    step lr along the orthogonalised gradient and is projected back to |w|_F = radius.

    Three library calls: X0 = g / (|g| + eps) (muonh_normalize), U = Newton-Schulz(X0) in
    place (muonh_newton_schulz), w = radius (w - lr radius U/|U|) / |w - lr radius U/|U||
    (muonh_apply)."""
    partials = _muonh_partials(w.device)
    x = muonh_normalize(g, eps=eps, partials=partials)
    muonh_newton_schulz(x, steps, coeffs)
    return muonh_apply(w, x, lr, radius, partials=partials)
