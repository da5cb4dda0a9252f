"""Python binding of ``libdt.so``, the GB300 conditional draft-tree builder.

Argument marshalling only: every step of a round runs in the library's CUDA
kernels. PyTorch provides device memory and streams. The functions mirror the
C ABI of ``include/dt.h`` (same names without the ``dt_`` prefix) and take
torch tensors where the C ABI takes pointers. When ``libdt.so`` is missing,
every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdt.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA = 0, -1, -2, -3
ERR_NONFINITE, ERR_TIMEOUT, ERR_BAD_TEMPERATURE = -4, -5, -6
F32, BF16 = 0, 1
NUM_PHASE_EVENTS = 4
OPT_TEST_BARRIER_TIMEOUT = 2  # dt_options.flags: failure-detection test hook
OPT_MARGINAL = 8             # dt_options.flags: marginal (path-independent) scores
OPT_STAGE_HOST_LOGITS = 16   # dt_options.flags: copy mapped host logits instead of reading in place
MAX_SPEC = 16

# every symbol include/dt.h declares
EXPORTS = ("dt_abi_version", "dt_status_string", "dt_prepared_bytes", "dt_prepare_weights",
           "dt_workspace_bytes", "dt_build_trees", "dt_host_workspace_bytes",
           "dt_build_trees_host", "dt_select_topm_noalloc", "dt_kernel_launches",
           "dt_chain_prepared_bytes", "dt_prepare_chain", "dt_chain_workspace_bytes",
           "dt_chain_kernel_launches", "dt_decode_chains", "dt_tree_positions",
           "dt_tree_attention", "dt_adaptive_budget", "dt_mapped_host_pointer")
NOALLOC_SCRATCH_BYTES = 8 << 20


class DtDims(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("V", "d", "d_s", "r", "D", "M", "k", "N", "batch")]


class DtWeights(C.Structure):
    _fields_ = [("E", C.c_void_p), ("W_ih", C.c_void_p), ("W_hh", C.c_void_p),
                ("b_ih", C.c_void_p), ("b_hh", C.c_void_p), ("W1", C.c_void_p),
                ("W2", C.c_void_p), ("wdtype", C.c_int)]


class DtTreeOut(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tokens", "parents", "depths", "scores", "mask",
                                           "topm", "status")]


class DtOptions(C.Structure):
    _fields_ = [("spec_width", C.c_int), ("phase_events", C.POINTER(C.c_void_p)),
                ("flags", C.c_int)]


class DtError(RuntimeError):
    pass


_lib = None


def lib():
    """Load libdt.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise DtError(f"{LIB_PATH} is not built; run conditional_draft_tree_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        L.dt_abi_version.restype = C.c_int
        L.dt_status_string.restype = C.c_char_p
        L.dt_status_string.argtypes = [C.c_int]
        L.dt_prepared_bytes.restype = C.c_size_t
        L.dt_prepared_bytes.argtypes = [C.POINTER(DtDims)]
        L.dt_prepare_weights.argtypes = [C.POINTER(DtDims), C.POINTER(DtWeights), C.c_void_p,
                                         C.c_size_t, C.c_void_p]
        L.dt_workspace_bytes.restype = C.c_size_t
        L.dt_workspace_bytes.argtypes = [C.POINTER(DtDims), C.POINTER(DtOptions)]
        L.dt_host_workspace_bytes.restype = C.c_size_t
        L.dt_host_workspace_bytes.argtypes = [C.POINTER(DtDims), C.POINTER(DtOptions)]
        L.dt_kernel_launches.restype = C.c_int
        L.dt_kernel_launches.argtypes = [C.POINTER(DtDims), C.c_int, C.POINTER(DtOptions)]
        sig = [C.POINTER(DtDims), C.POINTER(DtWeights), C.c_void_p, C.c_void_p, C.c_void_p,
               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
               C.POINTER(DtTreeOut), C.POINTER(DtOptions), C.c_void_p]
        L.dt_build_trees.argtypes = sig
        L.dt_build_trees_host.argtypes = sig
        L.dt_mapped_host_pointer.restype = C.c_void_p
        L.dt_mapped_host_pointer.argtypes = [C.c_void_p, C.c_size_t]
        L.dt_select_topm_noalloc.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                             C.c_void_p, C.c_void_p, C.c_void_p]
        L.dt_chain_prepared_bytes.restype = C.c_size_t
        L.dt_chain_prepared_bytes.argtypes = [C.POINTER(DtDims)]
        L.dt_prepare_chain.argtypes = [C.POINTER(DtDims), C.POINTER(DtWeights), C.c_void_p,
                                       C.c_size_t, C.c_void_p]
        L.dt_chain_workspace_bytes.restype = C.c_size_t
        L.dt_chain_workspace_bytes.argtypes = [C.POINTER(DtDims)]
        L.dt_chain_kernel_launches.restype = C.c_int
        L.dt_chain_kernel_launches.argtypes = [C.POINTER(DtDims)]
        L.dt_decode_chains.argtypes = [C.POINTER(DtDims), C.POINTER(DtWeights)] + \
            [C.c_void_p] * 9 + [C.c_size_t] + [C.c_void_p] * 4
        L.dt_adaptive_budget.argtypes = [C.POINTER(DtTreeOut), C.c_int, C.c_int, C.c_double,
                                         C.c_double, C.c_void_p, C.c_void_p]
        L.dt_tree_positions.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                        C.c_void_p]
        L.dt_tree_attention.argtypes = [C.c_void_p] * 5 + [C.c_int] * 6 + [C.c_float, C.c_void_p,
                                                                          C.c_void_p]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().dt_status_string(int(code)).decode()


def abi_version() -> int:
    return lib().dt_abi_version()


def _check(rc: int, what: str):
    if rc != OK:
        raise DtError(f"{what}: {status_string(rc)} ({rc})")


def dims_of(V, d, d_s, r, D, M, k, N, batch) -> DtDims:
    return DtDims(V, d, d_s, r, D, M, k, N, batch)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def options(spec_width: int = 0, events=None, flags: int = 0) -> DtOptions:
    """Build a dt_options; ``events``: DT_NUM_PHASE_EVENTS torch.cuda.Event or None;
    ``flags``: OPT_* bits."""
    o = DtOptions(spec_width, None, flags)
    if events is not None:
        arr = (C.c_void_p * NUM_PHASE_EVENTS)(*[e.cuda_event for e in events])
        o.phase_events = C.cast(arr, C.POINTER(C.c_void_p))
        o._keep = arr
    return o


@dataclass
class DeviceWeights:
    """Domino head weights on the device (see dt_weights in include/dt.h)."""
    E: torch.Tensor
    W_ih: torch.Tensor
    W_hh: torch.Tensor
    W1: torch.Tensor
    W2: torch.Tensor
    b_ih: torch.Tensor | None = None
    b_hh: torch.Tensor | None = None

    @property
    def wdtype(self) -> int:
        return BF16 if self.E.dtype in (torch.int16, torch.uint16, torch.bfloat16) else F32

    def struct(self) -> DtWeights:
        return DtWeights(_ptr(self.E), _ptr(self.W_ih), _ptr(self.W_hh), _ptr(self.b_ih),
                         _ptr(self.b_hh), _ptr(self.W1), _ptr(self.W2), self.wdtype)


def prepared_bytes(dims: DtDims) -> int:
    return lib().dt_prepared_bytes(C.byref(dims))


def prepare_weights(dims: DtDims, w: DeviceWeights, prepared: torch.Tensor, stream=None):
    ws = w.struct()
    _check(lib().dt_prepare_weights(C.byref(dims), C.byref(ws), prepared.data_ptr(),
                                    prepared.numel() * prepared.element_size(), _stream(stream)),
           "dt_prepare_weights")


def workspace_bytes(dims: DtDims, opt: DtOptions | None = None) -> int:
    return lib().dt_workspace_bytes(C.byref(dims), C.byref(opt) if opt else None)


def kernel_launches(dims: DtDims, wdtype: int, opt: DtOptions | None = None) -> int:
    """Kernels one build_trees call launches (see dt_kernel_launches)."""
    return lib().dt_kernel_launches(C.byref(dims), int(wdtype), C.byref(opt) if opt else None)


def host_workspace_bytes(dims: DtDims, opt: DtOptions | None = None) -> int:
    return lib().dt_host_workspace_bytes(C.byref(dims), C.byref(opt) if opt else None)


def alloc_outputs(dims: DtDims, device, mask=True, topm=True, pin=False):
    """Output tensors of dt_tree_out (device, or pinned host with device='cpu', pin=True)."""
    n1 = dims.N + 1
    kw = dict(device=device, pin_memory=pin) if pin else dict(device=device)
    out = dict(tokens=torch.empty((dims.batch, n1), dtype=torch.int32, **kw),
               parents=torch.empty((dims.batch, n1), dtype=torch.int32, **kw),
               depths=torch.empty((dims.batch, n1), dtype=torch.int32, **kw),
               scores=torch.empty((dims.batch, n1), dtype=torch.float32, **kw),
               status=torch.empty((dims.batch,), dtype=torch.int32, **kw))
    out["mask"] = torch.empty((dims.batch, n1, n1), dtype=torch.uint8, **kw) if mask else None
    out["topm"] = (torch.empty((dims.batch, dims.D, dims.M), dtype=torch.int32, **kw)
                   if topm else None)
    return out


def _out_struct(out) -> DtTreeOut:
    return DtTreeOut(*[_ptr(out.get(n)) for n in ("tokens", "parents", "depths", "scores",
                                                  "mask", "topm", "status")])


def build_trees(dims: DtDims, w: DeviceWeights, prepared, base_logits, H, state0, anchor_tok,
                temperature, workspace, out, opt: DtOptions | None = None, stream=None):
    """Enqueue one round on device tensors (dt_build_trees). With OPT_MARGINAL in
    ``opt.flags``, ``w``, ``prepared``, ``H`` and ``state0`` may be None."""
    ws = w.struct() if w is not None else None
    o = _out_struct(out)
    _check(lib().dt_build_trees(C.byref(dims), C.byref(ws) if ws else None, _ptr(prepared),
                                _ptr(base_logits),
                                _ptr(H), _ptr(state0), _ptr(anchor_tok), _ptr(temperature),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                C.byref(o), C.byref(opt) if opt else None, _stream(stream)),
           "dt_build_trees")


def build_trees_host(dims: DtDims, w: DeviceWeights, prepared, base_logits, H, state0,
                     anchor_tok, temperature, workspace, host_out, opt: DtOptions | None = None,
                     stream=None):
    """Enqueue one round on HOST input/output tensors (dt_build_trees_host). Synchronise
    the stream before reading ``host_out``."""
    ws = w.struct() if w is not None else None
    o = _out_struct(host_out)
    _check(lib().dt_build_trees_host(C.byref(dims), C.byref(ws) if ws else None, _ptr(prepared),
                                     _ptr(base_logits), _ptr(H), _ptr(state0), _ptr(anchor_tok),
                                     _ptr(temperature), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), C.byref(o),
                                     C.byref(opt) if opt else None, _stream(stream)),
           "dt_build_trees_host")


def mapped_host_pointer(t) -> int | None:
    """dt_mapped_host_pointer for a host tensor's whole storage extent: the
    device address kernels can read it through in place, or None."""
    return lib().dt_mapped_host_pointer(_ptr(t), t.numel() * t.element_size()) or None


def select_topm_noalloc(base_logits, M: int, topm, status, stream=None) -> int:
    """dt_select_topm_noalloc on device tensors: base_logits [batch][D][V] fp32,
    topm [batch][D][M] int32 and status [batch] int32 outputs. Allocates no
    device memory (the library's static scratch is used; see include/dt.h).
    Returns the C status code."""
    if base_logits.dim() != 3 or base_logits.dtype != torch.float32 or \
            not base_logits.is_contiguous() or not base_logits.is_cuda:
        raise ValueError("base_logits must be a contiguous [batch][D][V] float32 CUDA tensor")
    batch, D, V = base_logits.shape
    dev = base_logits.device
    if topm.shape != (batch, D, int(M)) or topm.dtype != torch.int32 or \
            not topm.is_contiguous() or topm.device != dev:
        raise ValueError("topm must be a contiguous [batch][D][M] int32 tensor on base_logits' device")
    if status.shape != (batch,) or status.dtype != torch.int32 or \
            not status.is_contiguous() or status.device != dev:
        raise ValueError("status must be a contiguous [batch] int32 tensor on base_logits' device")
    with torch.cuda.device(dev):
        return lib().dt_select_topm_noalloc(_ptr(base_logits), batch, D, V, int(M), _ptr(topm),
                                            _ptr(status), _stream(stream))


class TreeBuilder:
    """Holds device weights, the prepared table and a workspace for one shape.

    ``TreeBuilder.from_numpy(workload)`` copies a host workload's weights to the
    device and prepares them; ``run(...)`` builds one round on device tensors."""

    def __init__(self, dims: DtDims, weights: DeviceWeights, spec_width: int = 0,
                 device="cuda", flags: int = 0):
        self.dims = dims
        self.w = weights
        self.device = torch.device(device)
        self.opt = options(spec_width, flags=flags)
        nbytes = prepared_bytes(dims)
        if nbytes == 0:
            raise DtError("invalid dims")
        self.prepared = torch.empty(nbytes // 4, dtype=torch.float32, device=self.device)
        prepare_weights(dims, weights, self.prepared)
        wsb = workspace_bytes(dims, self.opt)
        if wsb == 0:
            raise DtError("dt_workspace_bytes failed (invalid dims or unsupported device)")
        self.workspace = torch.empty(wsb, dtype=torch.uint8, device=self.device)

    @staticmethod
    def weights_from_numpy(wl, device="cuda") -> DeviceWeights:
        import numpy as np

        def t(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            return torch.from_numpy(a).to(device)
        return DeviceWeights(E=t(wl.E), W_ih=t(wl.W_ih), W_hh=t(wl.W_hh), W1=t(wl.W1),
                             W2=t(wl.W2), b_ih=t(wl.b_ih), b_hh=t(wl.b_hh))

    @classmethod
    def from_numpy(cls, wl, spec_width: int = 0, device="cuda", batch=None, flags: int = 0):
        dims = dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N,
                       wl.batch if batch is None else batch)
        return cls(dims, cls.weights_from_numpy(wl, device), spec_width, device, flags)

    def run(self, base_logits, H, state0, anchor_tok, temperature=None, out=None, stream=None,
            opt=None):
        if out is None:
            out = alloc_outputs(self.dims, self.device)
        build_trees(self.dims, self.w, self.prepared, base_logits, H, state0, anchor_tok,
                    temperature, self.workspace, out, opt or self.opt, stream)
        return out

    def inputs_to_device(self, wl):
        import numpy as np
        f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(self.device)
        return dict(base_logits=f(wl.base_logits, np.float32), H=f(wl.H, np.float32),
                    state0=f(wl.state0, np.float32), anchor_tok=f(wl.anchor, np.int32),
                    temperature=f(wl.temperature, np.float32))


class MarginalTreeBuilder:
    """Workspace for marginal-score trees (OPT_MARGINAL) of one shape: no
    weights, no GRU state; ``run(base_logits, anchor_tok, temperature)`` builds
    one round on device tensors. ``dims`` keeps d, d_s and r only for the
    shape checks of the C ABI (any valid values)."""

    def __init__(self, dims: DtDims, device="cuda", spec_width: int = 0):
        self.dims = dims
        self.device = torch.device(device)
        self.opt = options(spec_width, flags=OPT_MARGINAL)
        wsb = workspace_bytes(dims, self.opt)
        if wsb == 0:
            raise DtError("dt_workspace_bytes failed (invalid dims or unsupported device)")
        self.workspace = torch.empty(wsb, dtype=torch.uint8, device=self.device)

    @classmethod
    def from_workload(cls, wl, device="cuda", batch=None):
        return cls(dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N,
                           wl.batch if batch is None else batch), device)

    def run(self, base_logits, anchor_tok, temperature=None, out=None, stream=None, opt=None):
        if out is None:
            out = alloc_outputs(self.dims, self.device)
        build_trees(self.dims, None, None, base_logits, None, None, anchor_tok, temperature,
                    self.workspace, out, opt or self.opt, stream)
        return out

    def inputs_to_device(self, wl):
        import numpy as np
        f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(self.device)
        return dict(base_logits=f(wl.base_logits, np.float32), anchor_tok=f(wl.anchor, np.int32),
                    temperature=f(wl.temperature, np.float32))



# ------------------------------------------------------------ chain decoding

def chain_prepared_bytes(dims: DtDims) -> int:
    return lib().dt_chain_prepared_bytes(C.byref(dims))


def prepare_chain(dims: DtDims, w: DeviceWeights, chain_prepared: torch.Tensor, stream=None):
    """dt_prepare_chain: the weight tiles of the chain decoder's tensor-core products."""
    ws = w.struct()
    _check(lib().dt_prepare_chain(C.byref(dims), C.byref(ws), chain_prepared.data_ptr(),
                                  chain_prepared.numel() * chain_prepared.element_size(),
                                  _stream(stream)), "dt_prepare_chain")


def chain_workspace_bytes(dims: DtDims) -> int:
    return lib().dt_chain_workspace_bytes(C.byref(dims))


def chain_kernel_launches(dims: DtDims) -> int:
    return lib().dt_chain_kernel_launches(C.byref(dims))


def decode_chains(dims: DtDims, w: DeviceWeights, prepared, chain_prepared, base_logits, H,
                  state0, anchor_tok, temperature, uniforms, workspace, tokens, logprobs, status,
                  stream=None):
    """Enqueue one chain-decoding round on device tensors (dt_decode_chains)."""
    ws = w.struct()
    _check(lib().dt_decode_chains(C.byref(dims), C.byref(ws), _ptr(prepared), _ptr(chain_prepared),
                                  _ptr(base_logits), _ptr(H), _ptr(state0), _ptr(anchor_tok),
                                  _ptr(temperature), _ptr(uniforms), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _ptr(tokens),
                                  _ptr(logprobs), _ptr(status), _stream(stream)),
           "dt_decode_chains")


class ChainDecoder:
    """Device weights, both prepared tables and a workspace for Domino chain
    decoding of one shape (bf16 weights). ``run(...)`` decodes one round:
    D draft tokens and their log-probabilities per request."""

    def __init__(self, dims: DtDims, weights: DeviceWeights, device="cuda"):
        self.dims = dims
        self.w = weights
        self.device = torch.device(device)
        nbytes = prepared_bytes(dims)
        cbytes = chain_prepared_bytes(dims)
        if nbytes == 0 or cbytes == 0:
            raise DtError("invalid dims")
        self.prepared = torch.empty(nbytes // 4, dtype=torch.float32, device=self.device)
        prepare_weights(dims, weights, self.prepared)
        self.chain_prepared = torch.empty(cbytes, dtype=torch.uint8, device=self.device)
        prepare_chain(dims, weights, self.chain_prepared)
        wsb = chain_workspace_bytes(dims)
        if wsb == 0:
            raise DtError("dt_chain_workspace_bytes failed (invalid dims or unsupported device)")
        self.workspace = torch.empty(wsb, dtype=torch.uint8, device=self.device)

    @classmethod
    def from_numpy(cls, wl, device="cuda", batch=None):
        dims = dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N,
                       wl.batch if batch is None else batch)
        return cls(dims, TreeBuilder.weights_from_numpy(wl, device), device)

    def alloc_outputs(self):
        B, D = self.dims.batch, self.dims.D
        return dict(tokens=torch.empty((B, D), dtype=torch.int32, device=self.device),
                    logprobs=torch.empty((B, D), dtype=torch.float32, device=self.device),
                    status=torch.empty((B,), dtype=torch.int32, device=self.device))

    def run(self, base_logits, H, state0, anchor_tok, temperature=None, uniforms=None, out=None,
            stream=None):
        if out is None:
            out = self.alloc_outputs()
        decode_chains(self.dims, self.w, self.prepared, self.chain_prepared, base_logits, H,
                      state0, anchor_tok, temperature, uniforms, self.workspace, out["tokens"],
                      out["logprobs"], out["status"], stream)
        return out

    def inputs_to_device(self, wl, uniforms=None):
        import numpy as np
        f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(self.device)
        d = dict(base_logits=f(wl.base_logits, np.float32), H=f(wl.H, np.float32),
                 state0=f(wl.state0, np.float32), anchor_tok=f(wl.anchor, np.int32),
                 temperature=f(wl.temperature, np.float32))
        if uniforms is not None:
            d["uniforms"] = f(uniforms, np.float32)
        return d



# ------------------------------------------------ verify-side consumption

def tree_positions(depths, prefix_len, out=None, stream=None):
    """dt_tree_positions on device tensors: depths [batch][n1] int32, prefix_len
    [batch] int32 -> position ids [batch][n1] int32."""
    batch, n1 = depths.shape
    if out is None:
        out = torch.empty_like(depths)
    _check(lib().dt_tree_positions(_ptr(depths), _ptr(prefix_len), batch, n1, _ptr(out),
                                   _stream(stream)), "dt_tree_positions")
    return out


def tree_attention(q, k, v, mask, prefix_len, scale=None, out=None, stream=None):
    """dt_tree_attention on device tensors: q [batch][H][n1][dh], k and v
    [batch][Hkv][P + n1][dh] (bf16, or int16/uint16 holding bf16 bits), mask
    [batch][n1][n1] uint8, prefix_len [batch] int32 -> fp32 [batch][H][n1][dh]."""
    batch, H, n1, dh = q.shape
    Hkv, L = k.shape[1], k.shape[2]
    if scale is None:
        scale = dh ** -0.5
    if out is None:
        out = torch.empty((batch, H, n1, dh), dtype=torch.float32, device=q.device)
    _check(lib().dt_tree_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(prefix_len), batch,
                                   H, Hkv, n1, L - n1, dh, float(scale), _ptr(out),
                                   _stream(stream)), "dt_tree_attention")
    return out



def adaptive_budget(out: dict, N: int, c_fixed: float, c_node: float, counts=None, stream=None):
    """dt_adaptive_budget: cut the trees of ``out`` (alloc_outputs layout, on
    the device) in place by the cost-aware rule; returns counts [batch] int32."""
    batch = out["tokens"].shape[0]
    if counts is None:
        counts = torch.empty(batch, dtype=torch.int32, device=out["tokens"].device)
    o = _out_struct(out)
    _check(lib().dt_adaptive_budget(C.byref(o), batch, int(N), float(c_fixed), float(c_node),
                                    _ptr(counts), _stream(stream)), "dt_adaptive_budget")
    return counts
