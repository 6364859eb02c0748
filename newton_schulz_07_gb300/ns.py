"""PyTorch-facing binding of the C ABI: argument marshalling only.

Every step of the computation runs in the CUDA library; PyTorch supplies the
device memory and the current stream.  Names follow the C entry points.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)
DEFAULT_EPS = 1e-7


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _shape3(t):
    if t.dim() == 2:
        return 1, t.shape[0], t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2]
    raise ValueError(f"expected a 2-D matrix or a 3-D stack, got shape {tuple(t.shape)}")


def _check_bf16(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(batch: int, rows: int, cols: int) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_workspace_size(batch, rows, cols, ctypes.byref(n)), "muon_ns_workspace_size")
    return n.value


def workspace_region(batch: int, rows: int, cols: int, region: int) -> tuple[int, int]:
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_workspace_region(batch, rows, cols, region, ctypes.byref(off), ctypes.byref(nb)),
               "muon_ns_workspace_region")
    return off.value, nb.value


def alloc_workspace(batch: int, rows: int, cols: int, device=None) -> torch.Tensor:
    """A uint8 device buffer of muon_ns_workspace_size() bytes (256-byte aligned)."""
    return torch.empty(max(workspace_size(batch, rows, cols), 1), dtype=torch.uint8, device=device or "cuda")


def _coeffs(coeffs):
    a = (ctypes.c_float * 3)(*[float(v) for v in coeffs])
    return ctypes.cast(a, ctypes.POINTER(ctypes.c_float))


def muon_ns(G: torch.Tensor, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS,
            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Batched quintic Newton–Schulz of a bf16 matrix or (batch, rows, cols) stack.

    With `workspace` (from alloc_workspace) the call goes through muon_ns_ws;
    otherwise through muon_ns and the library's cached workspace.  `out` may be G.
    """
    _check_bf16(G, "G")
    b, r, c = _shape3(G)
    if out is None:
        out = torch.empty_like(G)
    _check_bf16(out, "out")
    if out.shape != G.shape or out.device != G.device:
        raise ValueError("out must match G in shape and device")
    L = _lib.lib()
    cf = _coeffs(coeffs)
    with torch.cuda.device(G.device):
        st = _stream(G.device)
        if workspace is not None:
            if workspace.device != G.device:
                raise ValueError("workspace must be on G's device")
            s = L.muon_ns_ws(_ptr(G), _ptr(out), b, r, c, int(steps), cf, float(eps),
                             _ptr(workspace), workspace.numel() * workspace.element_size(), st)
            _lib.check(s, "muon_ns_ws")
        else:
            _lib.check(L.muon_ns(_ptr(G), _ptr(out), b, r, c, int(steps), cf, float(eps), st), "muon_ns")
    return out


def muon_ns_normalize(G: torch.Tensor, workspace: torch.Tensor, eps: float = DEFAULT_EPS,
                      X: torch.Tensor | None = None, norms_only: bool = False):
    """X = G / (||G||_F + eps); the norms go to the workspace's NORMS region.
    With norms_only=True only the norm kernel runs and None is returned."""
    _check_bf16(G, "G")
    b, r, c = _shape3(G)
    if norms_only:
        X = None
    elif X is None:
        X = torch.empty_like(G)
    with torch.cuda.device(G.device):
        _lib.check(_lib.lib().muon_ns_normalize(_ptr(G), _ptr(X), b, r, c, float(eps), _ptr(workspace),
                                                workspace.numel(), _stream(G.device)), "muon_ns_normalize")
    return X


def muon_ns_gram(X: torch.Tensor, A: torch.Tensor | None = None, device_error: torch.Tensor | None = None,
                 norms: torch.Tensor | None = None, eps: float = DEFAULT_EPS, half: bool = False):
    """A = X X^T (X^T X for tall X); with `norms` (fp32 [batch]) X is unscaled
    and the Gram of X / (norms + eps) is computed.  `half`: A stored half, as
    whole calls keep it (diagonal 256-blocks whole, the lower triangle
    elsewhere; MUON_NS_HALF)."""
    _check_bf16(X, "X")
    b, r, c = _shape3(X)
    m = min(r, c)
    if A is None:
        A = torch.empty((b, m, m) if X.dim() == 3 else (m, m), dtype=torch.bfloat16, device=X.device)
    with torch.cuda.device(X.device):
        _lib.check(_lib.lib().muon_ns_gram_ex(_ptr(X), _ptr(A), b, r, c, _ptr(norms), float(eps),
                                              _lib.HALF if half else 0, _ptr(device_error), _stream(X.device)),
                   "muon_ns_gram")
    return A


def muon_ns_poly(A: torch.Tensor, b: float, c: float, B: torch.Tensor | None = None,
                 diag: torch.Tensor | None = None, device_error: torch.Tensor | None = None, half: bool = False):
    """B = b A + c A A.  With `diag` (fp32, batch*m elements) B's diagonal goes
    there in fp32 and B's stored diagonal is zero.  `half`: A read and B
    written in half storage."""
    _check_bf16(A, "A")
    bt, m, m2 = _shape3(A)
    if m != m2:
        raise ValueError("A must be square")
    if diag is not None and (diag.dtype != torch.float32 or diag.numel() != bt * m or not diag.is_contiguous()):
        raise ValueError("diag must be a contiguous float32 tensor of batch * m elements")
    B = torch.empty_like(A) if B is None else B
    with torch.cuda.device(A.device):
        _lib.check(_lib.lib().muon_ns_poly_ex(_ptr(A), _ptr(B), _ptr(diag), bt, m, float(b), float(c),
                                              _lib.HALF if half else 0, _ptr(device_error), _stream(A.device)),
                   "muon_ns_poly")
    return B


def muon_ns_update(X: torch.Tensor, B: torch.Tensor, a: float, Xn: torch.Tensor | None = None,
                   diag: torch.Tensor | None = None, device_error: torch.Tensor | None = None,
                   norms: torch.Tensor | None = None, eps: float = DEFAULT_EPS, half: bool = False):
    """X' = a X + B X (X' = a X + X B for tall X).  With `diag` from
    muon_ns_poly, B = diag(D) + B_stored.  `half`: B read in half storage."""
    _check_bf16(X, "X")
    _check_bf16(B, "B")
    bt, r, c = _shape3(X)
    if diag is not None and (diag.dtype != torch.float32 or diag.numel() != bt * min(r, c)
                             or not diag.is_contiguous()):
        raise ValueError("diag must be a contiguous float32 tensor of batch * min(rows, cols) elements")
    Xn = torch.empty_like(X) if Xn is None else Xn
    with torch.cuda.device(X.device):
        _lib.check(_lib.lib().muon_ns_update_ex(_ptr(X), _ptr(B), _ptr(diag), _ptr(Xn), bt, r, c, float(a),
                                                _ptr(norms), float(eps), _lib.HALF if half else 0,
                                                _ptr(device_error), _stream(X.device)),
                   "muon_ns_update")
    return Xn


def read_error(workspace: torch.Tensor, clear: bool = False) -> int:
    v = ctypes.c_int(0)
    with torch.cuda.device(workspace.device):
        s = _lib.lib().muon_ns_read_error(_ptr(workspace), ctypes.byref(v), int(clear), _stream(workspace.device))
    if s not in (_lib.OK, _lib.ERR_TIMEOUT):
        _lib.check(s, "muon_ns_read_error")
    return v.value


def muon_ns_check(workspace: torch.Tensor, host_word: torch.Tensor) -> None:
    """Enqueue on the current stream a copy of the workspace's device error
    word into `host_word` (a pinned host int32 tensor of one element); no
    synchronisation, so it can be captured in a CUDA graph.  After the stream
    passes the copy, error_status(host_word.item()) gives the call's status."""
    if (not isinstance(host_word, torch.Tensor) or host_word.dtype != torch.int32 or host_word.is_cuda
            or host_word.numel() < 1 or not host_word.is_pinned()):
        raise TypeError("host_word must be a pinned host int32 tensor")
    with torch.cuda.device(workspace.device):
        _lib.check(_lib.lib().muon_ns_check(_ptr(workspace), _ptr(host_word), _stream(workspace.device)),
                   "muon_ns_check")


def error_status(word: int) -> int:
    """Status of a call from its device error word (see muon_ns_check)."""
    return _lib.ERR_TIMEOUT if int(word) & _lib.DEVERR_WAIT_TIMEOUT else _lib.OK


def host_chunk(batch: int, rows: int, cols: int, chunk: int = 0) -> int:
    """Largest chunk (matrices) muon_ns_host uses for this stack and `chunk`."""
    return _lib.lib().muon_ns_host_chunk(int(batch), int(rows), int(cols), int(chunk))


def host_plan(batch: int, rows: int, cols: int, chunk: int = 0) -> list:
    """Chunk sizes, in order, that muon_ns_host uses for this stack and `chunk`."""
    L = _lib.lib()
    n = L.muon_ns_host_plan(int(batch), int(rows), int(cols), int(chunk), None, 0)
    if n < 0:
        raise ValueError("invalid stack shape")
    arr = (ctypes.c_int * max(n, 1))()
    L.muon_ns_host_plan(int(batch), int(rows), int(cols), int(chunk), ctypes.cast(arr, ctypes.c_void_p), n)
    return list(arr[:n])


def set_wait_budget(cycles: int) -> None:
    """Budget of every bounded wait in the kernels, in SM clock cycles (0: the
    default, about 2 s).  A wait that runs out sets the device error word."""
    _lib.check(_lib.lib().muon_ns_set_wait_budget(int(cycles)), "muon_ns_set_wait_budget")


def inject_stall(enable: bool) -> None:
    """Host-side fault injection for tests: later whole calls of multi-matrix
    stacks wait for a completion that never comes, so their bounded waits run
    out and the device error word is set."""
    _lib.check(_lib.lib().muon_ns_inject_stall(int(bool(enable))), "muon_ns_inject_stall")


def launches_per_call(steps: int) -> int:
    return _lib.lib().muon_ns_launches_per_call(steps)


def muon_ns_normalize_static(G: torch.Tensor, eps: float = DEFAULT_EPS, X: torch.Tensor | None = None) -> torch.Tensor:
    """muon_ns_normalize without a workspace: for callers that cannot allocate
    device memory; its scratch is the library's 1 MiB static device array
    (see include/muon_ns.h for the size limit and the sharing rules)."""
    _check_bf16(G, "G")
    b, r, c = _shape3(G)
    X = torch.empty_like(G) if X is None else X
    with torch.cuda.device(G.device):
        _lib.check(_lib.lib().muon_ns_normalize_static(_ptr(G), _ptr(X), b, r, c, float(eps), _stream(G.device)),
                   "muon_ns_normalize_static")
    return X


def _stack_array(Gs, outs):
    arr = (_lib.MuonNSStack * max(len(Gs), 1))()
    for i, (G, o) in enumerate(zip(Gs, outs)):
        b, r, c = _shape3(G)
        arr[i] = _lib.MuonNSStack(G.data_ptr(), o.data_ptr(), b, r, c)
    return arr


def grouped_workspace_size(Gs) -> int:
    arr = _stack_array(Gs, Gs)
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_grouped_workspace_size(arr, len(Gs), ctypes.byref(n)),
               "muon_ns_grouped_workspace_size")
    return n.value


def muon_ns_grouped(Gs, outs=None, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS,
                    workspace: torch.Tensor | None = None):
    """NS of several stacks (a list of bf16 CUDA matrices or stacks, any shapes)
    in one call; returns the list of outputs (`outs[i]` may be `Gs[i]`)."""
    Gs = list(Gs)
    if not Gs:
        return []
    dev = Gs[0].device
    for G in Gs:
        _check_bf16(G, "G")
        if G.device != dev:
            raise ValueError("all stacks must be on one device")
    outs = [torch.empty_like(G) for G in Gs] if outs is None else list(outs)
    for G, o in zip(Gs, outs):
        _check_bf16(o, "out")
        if o.shape != G.shape or o.device != dev:
            raise ValueError("outs must match Gs")
    if workspace is None:
        workspace = torch.empty(max(grouped_workspace_size(Gs), 1), dtype=torch.uint8, device=dev)
    arr = _stack_array(Gs, outs)
    with torch.cuda.device(dev):
        _lib.check(_lib.lib().muon_ns_grouped(arr, len(Gs), int(steps), _coeffs(coeffs), float(eps),
                                              _ptr(workspace), workspace.numel(), _stream(dev)),
                   "muon_ns_grouped")
    return outs


def f32_workspace_size(batch: int, rows: int, cols: int) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_f32_workspace_size(batch, rows, cols, ctypes.byref(n)), "muon_ns_f32_workspace_size")
    return n.value


def f32_workspace_region(batch: int, rows: int, cols: int, region: int) -> tuple[int, int]:
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_f32_workspace_region(batch, rows, cols, region, ctypes.byref(off),
                                                       ctypes.byref(nb)), "muon_ns_f32_workspace_region")
    return off.value, nb.value


def muon_ns_f32(G: torch.Tensor, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS,
                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 Newton-Schulz of an fp32 matrix or (batch, rows, cols) stack (tf32
    tensor cores, fp32 storage); `out` may be G."""
    if not isinstance(G, torch.Tensor) or G.dtype != torch.float32 or not G.is_cuda or not G.is_contiguous():
        raise TypeError("G must be a contiguous CUDA float32 tensor")
    b, r, c = _shape3(G)
    out = torch.empty_like(G) if out is None else out
    if out.dtype != torch.float32 or out.shape != G.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor shaped like G")
    if workspace is None:
        workspace = torch.empty(max(f32_workspace_size(b, r, c), 1), dtype=torch.uint8, device=G.device)
    with torch.cuda.device(G.device):
        _lib.check(_lib.lib().muon_ns_ws_f32(_ptr(G), _ptr(out), b, r, c, int(steps), _coeffs(coeffs), float(eps),
                                             _ptr(workspace), workspace.numel(), _stream(G.device)), "muon_ns_ws_f32")
    return out


def host_workspace_size(batch: int, rows: int, cols: int, chunk: int = 0) -> int:
    """Device workspace bytes muon_ns_host needs (chunk <= 0: the default)."""
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_ns_host_workspace_size(int(batch), int(rows), int(cols), int(chunk), ctypes.byref(n)),
               "muon_ns_host_workspace_size")
    return n.value


def muon_ns_host(G: torch.Tensor, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS,
                 out: torch.Tensor | None = None, chunk: int = 0, workspace: torch.Tensor | None = None,
                 device=None, sync: bool = True) -> torch.Tensor:
    """NS of a bf16 matrix or stack held in host memory: the library uploads,
    orthogonalises and downloads it in chunks of `chunk` matrices, the copies
    overlapping the compute.  `out` (host, may be G) receives the result;
    with sync=False the caller synchronises the current stream of `device`
    before reading it.  Pin G and out (Tensor.pin_memory()) for overlap."""
    if not isinstance(G, torch.Tensor) or G.dtype != torch.bfloat16 or G.is_cuda or not G.is_contiguous():
        raise TypeError("G must be a contiguous host bfloat16 tensor")
    b, r, c = _shape3(G)
    if out is None:
        out = torch.empty_like(G, pin_memory=G.is_pinned())
    if out.dtype != torch.bfloat16 or out.is_cuda or out.shape != G.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous host bfloat16 tensor shaped like G")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if workspace is None:
        workspace = torch.empty(max(host_workspace_size(b, r, c, chunk), 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _lib.check(_lib.lib().muon_ns_host(_ptr(G), _ptr(out), b, r, c, int(steps), _coeffs(coeffs), float(eps),
                                           int(chunk), _ptr(workspace), workspace.numel(), _stream(dev)),
                   "muon_ns_host")
        if sync:
            torch.cuda.current_stream(dev).synchronize()
    return out


# ---------------------------------------------------------------- Muon step --

def _check_f32(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA float32 tensor")


def default_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows / cols)): the shape factor on the orthogonalised update."""
    return math.sqrt(max(1.0, rows / cols))


def _hparams(lr, momentum, weight_decay, scale, nesterov):
    return _lib.MuonStepHparams(float(lr), float(momentum), float(weight_decay), float(scale), int(bool(nesterov)))


def step_workspace_size(batch: int, rows: int, cols: int) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_step_workspace_size(batch, rows, cols, ctypes.byref(n)), "muon_step_workspace_size")
    return n.value


def muon_step(W: torch.Tensor, M: torch.Tensor, G: torch.Tensor, lr: float, momentum: float = 0.95,
              nesterov: bool = True, weight_decay: float = 0.0, scale: float | None = None, steps: int = 5,
              coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS, workspace: torch.Tensor | None = None) -> None:
    """One Muon step, in place on the fp32 master W and momentum M, for an
    fp32 gradient G (matrix or (batch, rows, cols) stack):
    M = mu M + G; U = G + mu M (Nesterov) or M; W = (1 - lr wd) W - lr scale NS(bf16(U)).
    `scale` defaults to sqrt(max(1, rows / cols))."""
    for t, n in ((W, "W"), (M, "M"), (G, "G")):
        _check_f32(t, n)
        if t.shape != W.shape or t.device != W.device:
            raise ValueError("W, M and G must have one shape and device")
    b, r, c = _shape3(W)
    hp = _hparams(lr, momentum, weight_decay, default_scale(r, c) if scale is None else scale, nesterov)
    if workspace is None:
        workspace = torch.empty(max(step_workspace_size(b, r, c), 1), dtype=torch.uint8, device=W.device)
    with torch.cuda.device(W.device):
        _lib.check(_lib.lib().muon_step_ws(_ptr(W), _ptr(M), _ptr(G), b, r, c, ctypes.byref(hp), int(steps),
                                           _coeffs(coeffs), float(eps), _ptr(workspace), workspace.numel(),
                                           _stream(W.device)), "muon_step_ws")


def muon_momentum(M: torch.Tensor, G: torch.Tensor, workspace: torch.Tensor, momentum: float = 0.95,
                  nesterov: bool = True, U: torch.Tensor | None = None) -> torch.Tensor:
    """The step's first kernel: M = mu M + G in place; returns the bf16 NS
    input U; ||U||_F goes to the (muon_ns_ws) workspace's NORMS region."""
    _check_f32(M, "M")
    _check_f32(G, "G")
    b, r, c = _shape3(M)
    U = torch.empty(M.shape, dtype=torch.bfloat16, device=M.device) if U is None else U
    _check_bf16(U, "U")
    with torch.cuda.device(M.device):
        _lib.check(_lib.lib().muon_momentum(_ptr(M), _ptr(G), _ptr(U), b, r, c, float(momentum), int(bool(nesterov)),
                                            _ptr(workspace), workspace.numel(), _stream(M.device)), "muon_momentum")
    return U


def muon_apply(W: torch.Tensor, O: torch.Tensor, lr: float, weight_decay: float = 0.0,
               scale: float | None = None) -> None:
    """The step's update alone: W = (1 - lr wd) W - lr scale O (O bf16, W's shape)."""
    _check_f32(W, "W")
    _check_bf16(O, "O")
    b, r, c = _shape3(W)
    hp = _hparams(lr, 0.0, weight_decay, default_scale(r, c) if scale is None else scale, False)
    with torch.cuda.device(W.device):
        _lib.check(_lib.lib().muon_apply(_ptr(W), _ptr(O), b, r, c, ctypes.byref(hp), _stream(W.device)),
                   "muon_apply")


def _step_stacks(groups):
    """ctypes array of muon_step_stack for a list of groups (dicts with W, M, G
    and the step's hyperparameters: lr, and optionally momentum, nesterov,
    weight_decay, scale)."""
    arr = (_lib.MuonStepStack * max(len(groups), 1))()
    for i, g in enumerate(groups):
        W, M, G = g["W"], g["M"], g["G"]
        for t, n in ((W, "W"), (M, "M"), (G, "G")):
            _check_f32(t, n)
            if t.shape != W.shape or t.device != W.device:
                raise ValueError("W, M and G of a group must have one shape and device")
        b, r, c = _shape3(W)
        scale = g.get("scale")
        hp = _hparams(g["lr"], g.get("momentum", 0.95), g.get("weight_decay", 0.0),
                      default_scale(r, c) if scale is None else scale, g.get("nesterov", True))
        arr[i] = _lib.MuonStepStack(W.data_ptr(), M.data_ptr(), G.data_ptr(), b, r, c, hp)
    return arr


def step_grouped_workspace_size(groups) -> int:
    arr = _step_stacks(groups)
    n = ctypes.c_size_t(0)
    _lib.check(_lib.lib().muon_step_grouped_workspace_size(arr, len(groups), ctypes.byref(n)),
               "muon_step_grouped_workspace_size")
    return n.value


def muon_step_grouped(groups, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS,
                      workspace: torch.Tensor | None = None) -> None:
    """One Muon step over several parameter groups in one call, in place on
    each group's W and M.  `groups` is a list of dicts with keys W, M, G (fp32
    CUDA tensors of one shape per group, all on one device) and lr, and
    optionally momentum (0.95), nesterov (True), weight_decay (0) and scale
    (sqrt(max(1, rows / cols)))."""
    groups = list(groups)
    if not groups:
        return
    dev = groups[0]["W"].device
    if any(g["W"].device != dev for g in groups):
        raise ValueError("all groups must be on one device")
    arr = _step_stacks(groups)
    if workspace is None:
        workspace = torch.empty(max(step_grouped_workspace_size(groups), 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _lib.check(_lib.lib().muon_step_grouped(arr, len(groups), int(steps), _coeffs(coeffs), float(eps),
                                                _ptr(workspace), workspace.numel(), _stream(dev)),
                   "muon_step_grouped")


def step_launches(steps: int) -> int:
    return _lib.lib().muon_step_launches(steps)
