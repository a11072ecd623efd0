"""Python binding of the GB300 Mamba2 SSD varlen prefill library (ctypes).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libssd_varlen.so, called through its C ABI (include/ssd_varlen.h).  PyTorch
only provides device memory and the current stream.  There is no CPU
fallback: if the library is missing the calls raise.

The functions keep the C names:
  ssd_varlen_workspace_size(dims)                 -> bytes
  ssd_varlen_count_chunks(cu_host, ncomp_host, Q) -> export rows
  ssd_varlen_plan(dims, cu_seqlens, num_computed, workspace) -> Plan
  ssd_varlen_forward(plan, inputs, outputs)
  ssd_varlen_status(plan)                          -> device error bits
  ssd_varlen_forward_path(plan, inputs, outputs)   -> (path, tile), no launch
  ssd_varlen_strerror(code)                        -> text
  ssd_varlen_forward_static(...)   (C only: forward without a caller workspace)
  ssd_varlen_decode(dims, cu_seqlens, io)        (decode / speculative-decode step)
  ssd_varlen_conv1d(dims, cu_seqlens, io)        (varlen causal conv1d with conv-state anchors)
  ssd_varlen_align_bite(start, end, total, align) (block-aligned prefill bite, host)
  ssd_varlen_gdn_forward(dims, cu_seqlens, io)   (gated delta rule prefill by chunks)
  ssd_varlen_check_slots(dims, init, final, block_table, err)  (slot-aliasing check, debug)
and ``run(...)`` wires a whole call from torch tensors (tests and bench use it).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libssd_varlen.so")

DTYPE_BF16 = 0
DTYPE_F32 = 1

DEVERR = {
    "CU_SEQLENS": 0x1, "NUM_COMPUTED": 0x2, "INIT_SLOT": 0x4, "FINAL_SLOT": 0x8,
    "BLOCK_SLOT": 0x10, "BLOCK_TABLE": 0x20, "TIMEOUT": 0x40, "INTERNAL": 0x80, "ALIAS": 0x100,
}
STATUS = {
    0: "OK", -1: "NULL", -2: "DIMS", -3: "CHUNK_SIZE", -4: "GROUPS", -5: "BLOCK_SIZE",
    -6: "DTYPE", -7: "ALIGN", -8: "WORKSPACE", -9: "PLAN", -10: "CUDA", -11: "UNSUPPORTED",
}
EXPORTED = ["ssd_varlen_workspace_size", "ssd_varlen_count_chunks", "ssd_varlen_plan",
            "ssd_varlen_forward", "ssd_varlen_status", "ssd_varlen_strerror",
            "ssd_varlen_forward_static", "ssd_varlen_decode", "ssd_varlen_conv1d",
            "ssd_varlen_align_bite", "ssd_varlen_gdn_forward", "ssd_varlen_check_slots",
            "ssd_varlen_forward_path"]
# enum ssd_path
PATH_TENSOR_CORE = 1
PATH_GENERAL = 2
PATH_TENSOR_CORE_PAIRED = 3
PATHS_TENSOR_CORE = (PATH_TENSOR_CORE, PATH_TENSOR_CORE_PAIRED)
# Size of the library-owned scratch array used by ssd_varlen_forward_static.
STATIC_SCRATCH_BYTES = 32 << 20

c_i32, c_i64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p


class ssd_dims(ctypes.Structure):
    _fields_ = [("T", c_i64), ("R", c_i32), ("H", c_i32), ("P", c_i32), ("N", c_i32),
                ("G", c_i32), ("chunk_size", c_i32), ("dtype", c_i32), ("num_slots", c_i32),
                ("block_size", c_i32), ("block_table_width", c_i32), ("reserved", c_i32)]


class ssd_plan(ctypes.Structure):
    _fields_ = [("dims", ssd_dims), ("workspace", c_vp), ("workspace_bytes", ctypes.c_size_t),
                ("cu_seqlens", c_vp), ("num_computed", c_vp), ("max_chunks", c_i64),
                ("max_segs", c_i64), ("seg_len", c_i32), ("flags", c_i32),
                ("magic", ctypes.c_uint64), ("stream", c_vp)]


class ssd_inputs(ctypes.Structure):
    _fields_ = [("x", c_vp), ("dt", c_vp), ("dt_bias", c_vp), ("A", c_vp), ("B", c_vp),
                ("C", c_vp), ("D", c_vp), ("z", c_vp), ("init_slots", c_vp),
                ("state_pool", c_vp)]


class ssd_outputs(ctypes.Structure):
    _fields_ = [("y", c_vp), ("final_states", c_vp), ("final_slots", c_vp),
                ("chunk_states", c_vp), ("block_table", c_vp)]


class ssd_decode_io(ctypes.Structure):
    _fields_ = [("x", c_vp), ("dt", c_vp), ("dt_bias", c_vp), ("A", c_vp), ("B", c_vp), ("C", c_vp),
                ("D", c_vp), ("z", c_vp), ("state_pool", c_vp), ("read_slots", c_vp),
                ("write_slots", c_vp), ("y", c_vp), ("device_err", c_vp)]


class ssd_conv_dims(ctypes.Structure):
    _fields_ = [("T", c_i64), ("R", c_i32), ("D", c_i32), ("W", c_i32), ("dtype", c_i32), ("num_slots", c_i32),
                ("silu", c_i32)]


class ssd_conv_io(ctypes.Structure):
    _fields_ = [("x", c_vp), ("weight", c_vp), ("bias", c_vp), ("conv_pool", c_vp), ("read_slots", c_vp),
                ("write_slots", c_vp), ("y", c_vp), ("device_err", c_vp)]


class ssd_gdn_dims(ctypes.Structure):
    _fields_ = [("T", c_i64), ("R", c_i32), ("Hk", c_i32), ("Hv", c_i32), ("K", c_i32), ("V", c_i32),
                ("chunk_size", c_i32), ("block_size", c_i32), ("block_table_width", c_i32), ("dtype", c_i32),
                ("num_slots", c_i32), ("l2norm", c_i32), ("scale", ctypes.c_float)]


class ssd_gdn_io(ctypes.Structure):
    _fields_ = [("q", c_vp), ("k", c_vp), ("v", c_vp), ("g", c_vp), ("beta", c_vp), ("num_computed", c_vp),
                ("state_pool", c_vp), ("init_slots", c_vp), ("final_slots", c_vp), ("block_table", c_vp),
                ("o", c_vp), ("final_states", c_vp), ("chunk_states", c_vp), ("device_err", c_vp)]


class SsdError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({ssd_varlen_strerror(code)})")
        self.code = code


_lib = None


def load_library():
    """Load libssd_varlen.so (built by build.py).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.ssd_varlen_workspace_size.argtypes = [ctypes.POINTER(ssd_dims)]
    lib.ssd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.ssd_varlen_count_chunks.argtypes = [c_vp, c_vp, c_i32, c_i32]
    lib.ssd_varlen_count_chunks.restype = c_i64
    lib.ssd_varlen_plan.argtypes = [ctypes.POINTER(ssd_dims), c_vp, c_vp, c_vp, ctypes.c_size_t,
                                    c_vp, ctypes.POINTER(ssd_plan)]
    lib.ssd_varlen_plan.restype = ctypes.c_int
    lib.ssd_varlen_forward.argtypes = [ctypes.POINTER(ssd_plan), ctypes.POINTER(ssd_inputs),
                                       ctypes.POINTER(ssd_outputs), c_vp]
    lib.ssd_varlen_forward.restype = ctypes.c_int
    lib.ssd_varlen_status.argtypes = [ctypes.POINTER(ssd_plan), ctypes.POINTER(ctypes.c_int)]
    lib.ssd_varlen_status.restype = ctypes.c_int
    lib.ssd_varlen_strerror.argtypes = [ctypes.c_int]
    lib.ssd_varlen_strerror.restype = ctypes.c_char_p
    lib.ssd_varlen_forward_static.argtypes = [ctypes.POINTER(ssd_dims), c_vp, c_vp,
                                              ctypes.POINTER(ssd_inputs), ctypes.POINTER(ssd_outputs),
                                              c_vp, ctypes.POINTER(ssd_plan)]
    lib.ssd_varlen_forward_static.restype = ctypes.c_int
    lib.ssd_varlen_decode.argtypes = [ctypes.POINTER(ssd_dims), c_vp, ctypes.POINTER(ssd_decode_io), c_vp]
    lib.ssd_varlen_decode.restype = ctypes.c_int
    lib.ssd_varlen_conv1d.argtypes = [ctypes.POINTER(ssd_conv_dims), c_vp, ctypes.POINTER(ssd_conv_io), c_vp]
    lib.ssd_varlen_conv1d.restype = ctypes.c_int
    lib.ssd_varlen_align_bite.argtypes = [c_i64, c_i64, c_i64, c_i32]
    lib.ssd_varlen_align_bite.restype = c_i64
    lib.ssd_varlen_gdn_forward.argtypes = [ctypes.POINTER(ssd_gdn_dims), c_vp, ctypes.POINTER(ssd_gdn_io), c_vp]
    lib.ssd_varlen_gdn_forward.restype = ctypes.c_int
    lib.ssd_varlen_check_slots.argtypes = [ctypes.POINTER(ssd_dims), c_vp, c_vp, c_vp, c_vp, c_vp]
    lib.ssd_varlen_check_slots.restype = ctypes.c_int
    lib.ssd_varlen_forward_path.argtypes = [ctypes.POINTER(ssd_plan), ctypes.POINTER(ssd_inputs),
                                            ctypes.POINTER(ssd_outputs), ctypes.POINTER(ctypes.c_int),
                                            ctypes.POINTER(ctypes.c_int)]
    lib.ssd_varlen_forward_path.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_dims(T, R, H, P, N, G, chunk_size, dtype, num_slots=0, block_size=0,
              block_table_width=0) -> ssd_dims:
    return ssd_dims(int(T), int(R), int(H), int(P), int(N), int(G), int(chunk_size), int(dtype),
                    int(num_slots), int(block_size), int(block_table_width), 0)


def ssd_varlen_strerror(code: int) -> str:
    return load_library().ssd_varlen_strerror(int(code)).decode()


def ssd_varlen_workspace_size(dims: ssd_dims) -> int:
    return int(load_library().ssd_varlen_workspace_size(ctypes.byref(dims)))


def ssd_varlen_count_chunks(cu_host, ncomp_host, chunk_size) -> int:
    import numpy as np
    cu = np.ascontiguousarray(cu_host, dtype=np.int32)
    nc = None if ncomp_host is None else np.ascontiguousarray(ncomp_host, dtype=np.int32)
    n = load_library().ssd_varlen_count_chunks(
        cu.ctypes.data_as(c_vp), None if nc is None else nc.ctypes.data_as(c_vp),
        cu.shape[0] - 1, int(chunk_size))
    if n < 0:
        raise SsdError(int(n), "ssd_varlen_count_chunks")
    return int(n)


def ssd_varlen_plan(dims: ssd_dims, cu_seqlens, num_computed, workspace, stream=None) -> ssd_plan:
    plan = ssd_plan()
    rc = load_library().ssd_varlen_plan(ctypes.byref(dims), _ptr(cu_seqlens), _ptr(num_computed),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream), ctypes.byref(plan))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_plan")
    return plan


def ssd_varlen_forward(plan: ssd_plan, inputs: ssd_inputs, outputs: ssd_outputs, stream=None):
    rc = load_library().ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(inputs),
                                           ctypes.byref(outputs), _stream(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_forward")


def ssd_varlen_status(plan: ssd_plan) -> int:
    v = ctypes.c_int(0)
    rc = load_library().ssd_varlen_status(ctypes.byref(plan), ctypes.byref(v))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_status")
    return int(v.value)


def ssd_varlen_forward_path(plan: ssd_plan, inputs: ssd_inputs, outputs: ssd_outputs):
    """(path, tile): the kernel path ssd_varlen_forward takes for these arguments
    (PATH_TENSOR_CORE_PAIRED, PATH_TENSOR_CORE or PATH_GENERAL) and its internal tile in tokens."""
    path, tile = ctypes.c_int(0), ctypes.c_int(0)
    rc = load_library().ssd_varlen_forward_path(ctypes.byref(plan), ctypes.byref(inputs),
                                                ctypes.byref(outputs), ctypes.byref(path),
                                                ctypes.byref(tile))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_forward_path")
    return int(path.value), int(tile.value)


def make_inputs(x, dt, dt_bias, A, B, C, D=None, z=None, init_slots=None, state_pool=None):
    return ssd_inputs(_ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                      _ptr(z), _ptr(init_slots), _ptr(state_pool))


def make_outputs(y, final_states=None, final_slots=None, chunk_states=None, block_table=None):
    return ssd_outputs(_ptr(y), _ptr(final_states), _ptr(final_slots), _ptr(chunk_states),
                       _ptr(block_table))


class Call:
    """One planned batch: the tensors, the plan and the pre-built argument structs."""

    def __init__(self, prob: dict, want_final=True, want_chunks=None, stream=None):
        import torch
        self.prob = prob
        x = prob["x"]
        dev = x.device
        T, H, P = x.shape
        N = prob["B"].shape[2]
        G = prob["B"].shape[1]
        R = prob["cu_seqlens"].shape[0] - 1
        Q = int(prob["chunk_size"])
        dtype = DTYPE_F32 if x.dtype == torch.float32 else DTYPE_BF16
        pool = prob.get("state_pool")
        bt = prob.get("block_table")
        self.dims = make_dims(T, R, H, P, N, G, Q, dtype,
                              num_slots=0 if pool is None else pool.shape[0],
                              block_size=int(prob.get("block_size") or 0),
                              block_table_width=0 if bt is None else bt.shape[1])
        self.workspace = torch.empty(ssd_varlen_workspace_size(self.dims), dtype=torch.uint8,
                                     device=dev)
        self.y = torch.empty_like(x)
        self.final_states = (torch.empty((R, H, P, N), dtype=torch.float32, device=dev)
                             if want_final and prob.get("final_dense", True) else None)
        export = prob.get("export_chunks") if want_chunks is None else want_chunks
        self.chunk_states = None
        if export:
            cu_h = prob["cu_seqlens"].cpu().numpy()
            nc = prob.get("num_computed")
            nrows = ssd_varlen_count_chunks(cu_h, None if nc is None else nc.cpu().numpy(), Q)
            self.chunk_states = torch.empty((max(nrows, 1), H, P, N), dtype=torch.float32,
                                            device=dev)
        self.inputs = make_inputs(x, prob["dt"], prob["dt_bias"], prob["A"], prob["B"],
                                  prob["C"], prob.get("D"), prob.get("z"),
                                  prob.get("init_slots"), pool)
        self.outputs = make_outputs(self.y, self.final_states, prob.get("final_slots"),
                                    self.chunk_states, bt)
        self.stream = stream
        self.plan = None

    def make_plan(self):
        self.plan = ssd_varlen_plan(self.dims, self.prob["cu_seqlens"],
                                    self.prob.get("num_computed"), self.workspace, self.stream)
        return self.plan

    def forward(self):
        ssd_varlen_forward(self.plan, self.inputs, self.outputs, self.stream)

    def __call__(self):
        self.make_plan()
        self.forward()
        return self

    def status(self) -> int:
        return ssd_varlen_status(self.plan)

    def path(self):
        """(path, tile) the forward of this call takes (plans first if needed)."""
        if self.plan is None:
            self.make_plan()
        return ssd_varlen_forward_path(self.plan, self.inputs, self.outputs)


def run(prob: dict, **kw) -> Call:
    """Plan and run one call on the current stream; returns the Call (outputs on it)."""
    return Call(prob, **kw)()


def ssd_varlen_decode(dims: ssd_dims, cu_seqlens, io: "ssd_decode_io", stream=None):
    rc = load_library().ssd_varlen_decode(ctypes.byref(dims), _ptr(cu_seqlens), ctypes.byref(io),
                                          _stream(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_decode")


class DecodeCall:
    """One decode / speculative-decode step over a problem from workloads.make_decode_problem:
    the output y and the device error word, and the pre-built argument structs."""

    def __init__(self, prob: dict, stream=None):
        import torch
        self.prob = prob
        x = prob["x"]
        T, H, P = x.shape
        G, N = prob["B"].shape[1], prob["B"].shape[2]
        R = prob["cu_seqlens"].shape[0] - 1
        dtype = DTYPE_F32 if x.dtype == torch.float32 else DTYPE_BF16
        pool = prob["state_pool"]
        self.dims = make_dims(T, R, H, P, N, G, 0, dtype, num_slots=pool.shape[0])
        self.y = torch.empty_like(x)
        self.err = torch.zeros(4, dtype=torch.int32, device=x.device)
        self.io = ssd_decode_io(_ptr(x), _ptr(prob["dt"]), _ptr(prob["dt_bias"]), _ptr(prob["A"]),
                                _ptr(prob["B"]), _ptr(prob["C"]), _ptr(prob.get("D")), _ptr(prob.get("z")),
                                _ptr(pool), _ptr(prob["read_slots"]), _ptr(prob.get("write_slots")),
                                _ptr(self.y), _ptr(self.err))
        self.stream = stream

    def __call__(self):
        ssd_varlen_decode(self.dims, self.prob["cu_seqlens"], self.io, self.stream)
        return self

    def status(self) -> int:
        """Device error bits of the calls so far (synchronises), then clears them."""
        v = int(self.err[0].item())
        self.err.zero_()
        return v


def run_decode(prob: dict, **kw) -> DecodeCall:
    """One decode step on the current stream; returns the DecodeCall (y on it, pool updated)."""
    return DecodeCall(prob, **kw)()



def ssd_varlen_conv1d(dims: ssd_conv_dims, cu_seqlens, io: ssd_conv_io, stream=None):
    rc = load_library().ssd_varlen_conv1d(ctypes.byref(dims), _ptr(cu_seqlens), ctypes.byref(io), _stream(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_conv1d")


class Conv1dCall:
    """One varlen causal conv1d over a problem from workloads.make_conv_problem: the
    output y and the device error word, and the pre-built argument structs."""

    def __init__(self, prob: dict, stream=None):
        import torch
        self.prob = prob
        x = prob["x"]
        T, D = x.shape
        W = prob["weight"].shape[1]
        R = prob["cu_seqlens"].shape[0] - 1
        pool = prob.get("conv_pool")
        self.dims = ssd_conv_dims(T, R, D, W, DTYPE_F32 if x.dtype == torch.float32 else DTYPE_BF16,
                                  0 if pool is None else pool.shape[0], 1 if prob.get("silu") else 0)
        self.y = torch.empty_like(x)
        self.err = torch.zeros(4, dtype=torch.int32, device=x.device)
        self.io = ssd_conv_io(_ptr(x), _ptr(prob["weight"]), _ptr(prob.get("bias")), _ptr(pool),
                              _ptr(prob.get("read_slots")), _ptr(prob.get("write_slots")), _ptr(self.y),
                              _ptr(self.err))
        self.stream = stream

    def __call__(self):
        ssd_varlen_conv1d(self.dims, self.prob["cu_seqlens"], self.io, self.stream)
        return self

    def status(self) -> int:
        v = int(self.err[0].item())
        self.err.zero_()
        return v


def run_conv1d(prob: dict, **kw) -> Conv1dCall:
    """One conv1d on the current stream; returns the Conv1dCall (y on it, conv states updated)."""
    return Conv1dCall(prob, **kw)()


def ssd_varlen_align_bite(start: int, end: int, total: int, align: int) -> int:
    """Where a proposed prefill bite [start, end) of a prompt ending at ``total`` should end."""
    r = int(load_library().ssd_varlen_align_bite(int(start), int(end), int(total), int(align)))
    if r < 0:
        raise SsdError(r, "ssd_varlen_align_bite")
    return r


GDN_CHUNK = 64  # the chunk length of the GDN kernel


def ssd_varlen_gdn_forward(dims: ssd_gdn_dims, cu_seqlens, io: ssd_gdn_io, stream=None):
    rc = load_library().ssd_varlen_gdn_forward(ctypes.byref(dims), _ptr(cu_seqlens), ctypes.byref(io),
                                                _stream(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_gdn_forward")


class GdnCall:
    """One GDN prefill over a problem from workloads.make_gdn_problem: outputs (o,
    final_states, chunk_states when asked), the device error word, and the pre-built
    argument structs (so a bench can call it repeatedly)."""

    def __init__(self, prob: dict, stream=None):
        import torch
        self.prob = prob
        q, v = prob["q"], prob["v"]
        T, Hk, K = q.shape
        Hv, V = v.shape[1], v.shape[2]
        R = prob["cu_seqlens"].shape[0] - 1
        pool = prob.get("state_pool")
        bt = prob.get("block_table")
        dev = q.device
        self.final_states = (torch.empty((R, Hv, K, V), dtype=torch.float32, device=dev)
                             if prob.get("final_dense", True) else None)
        self.chunk_states = None
        if prob.get("export_chunks"):
            nc = prob.get("num_computed")
            n = ssd_varlen_count_chunks(prob["cu_seqlens"].cpu().numpy(),
                                        None if nc is None else nc.cpu().numpy(), GDN_CHUNK)
            self.chunk_states = torch.empty((max(n, 1), Hv, K, V), dtype=torch.float32, device=dev)
        self.o = torch.empty_like(v)
        self.err = torch.zeros(4, dtype=torch.int32, device=dev)
        self.dims = ssd_gdn_dims(T, R, Hk, Hv, K, V, GDN_CHUNK, int(prob.get("block_size") or 0),
                                 0 if bt is None else bt.shape[1],
                                 DTYPE_F32 if q.dtype == torch.float32 else DTYPE_BF16,
                                 0 if pool is None else pool.shape[0], 1 if prob.get("l2norm") else 0,
                                 float(prob.get("scale") or 0.0))
        self.io = ssd_gdn_io(_ptr(q), _ptr(prob["k"]), _ptr(v), _ptr(prob["g"]), _ptr(prob["beta"]),
                             _ptr(prob.get("num_computed")), _ptr(pool), _ptr(prob.get("init_slots")),
                             _ptr(prob.get("final_slots")), _ptr(bt), _ptr(self.o), _ptr(self.final_states),
                             _ptr(self.chunk_states), _ptr(self.err))
        self.stream = stream

    def __call__(self):
        ssd_varlen_gdn_forward(self.dims, self.prob["cu_seqlens"], self.io, self.stream)
        return self

    def status(self) -> int:
        v = int(self.err[0].item())
        self.err.zero_()
        return v


def run_gdn(prob: dict, **kw) -> GdnCall:
    """One GDN prefill on the current stream; returns the GdnCall (outputs on it)."""
    return GdnCall(prob, **kw)()


def ssd_varlen_check_slots(R, init_slots=None, final_slots=None, block_table=None, stream=None) -> int:
    """Device check that no written slot is read or written twice; returns the
    device error bits (SSD_DEVERR_ALIAS when it finds one).  Synchronises."""
    import torch
    dev = next(t.device for t in (init_slots, final_slots, block_table) if t is not None)
    err = torch.zeros(4, dtype=torch.int32, device=dev)
    width = 0 if block_table is None else int(block_table.shape[1])
    dims = make_dims(0, R, 1, 1, 1, 1, 16, DTYPE_BF16, block_table_width=width)
    rc = load_library().ssd_varlen_check_slots(ctypes.byref(dims), _ptr(init_slots), _ptr(final_slots),
                                               _ptr(block_table), _ptr(err), _stream(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_varlen_check_slots")
    torch.cuda.synchronize(dev)
    return int(err[0].item())
