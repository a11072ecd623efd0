"""C-ABI library: loads, exports every declared symbol, host-side validation (CPU only).

No call here reaches the GPU: every argument error is caught by the host code
before any launch, so these run on a machine without a CUDA device.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import mamba2_ssd_varlen_gb300 as m
from oracle import checkpoints

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    return m.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd_varlen.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_varlen_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) == set(m.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_sizes_match_header(lib):
    # ssd_dims: int64 + 11 int32 = 56 bytes; the binding mirrors the header.
    assert ctypes.sizeof(m.ssd_dims) == 56
    assert ctypes.sizeof(m.ssd_inputs) == 10 * 8
    assert ctypes.sizeof(m.ssd_outputs) == 5 * 8
    assert ctypes.sizeof(m.ssd_decode_io) == 13 * 8


def _dims(**kw):
    base = dict(T=64, R=3, H=4, P=16, N=16, G=1, chunk_size=16, dtype=m.DTYPE_F32,
                num_slots=3, block_size=0, block_table_width=0)
    base.update(kw)
    return m.make_dims(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(chunk_size=17), -3), (dict(chunk_size=8), -3), (dict(chunk_size=512), -3),
    (dict(chunk_size=0), -3), (dict(G=3), -4), (dict(H=0), -2), (dict(R=0), -2),
    (dict(T=-1), -2), (dict(dtype=7), -6), (dict(block_size=24), -5),
    (dict(block_size=-16), -5), (dict(N=48), -11), (dict(P=512), -2),
])
def test_plan_rejects_bad_dims_before_launch(lib, kw, code):
    d = _dims(**kw)
    plan = m.ssd_plan()
    rc = lib.ssd_varlen_plan(ctypes.byref(d), ctypes.c_void_p(0x1000), None,
                             ctypes.c_void_p(0x2000), 1 << 20, None, ctypes.byref(plan))
    assert rc == code
    assert lib.ssd_varlen_workspace_size(ctypes.byref(d)) == 0


def test_plan_null_and_workspace_checks(lib):
    d = _dims()
    plan = m.ssd_plan()
    ws = lib.ssd_varlen_workspace_size(ctypes.byref(d))
    assert ws > 0 and ws % 256 == 0
    assert lib.ssd_varlen_plan(ctypes.byref(d), None, None, ctypes.c_void_p(0x2000), ws, None,
                               ctypes.byref(plan)) == -1
    assert lib.ssd_varlen_plan(ctypes.byref(d), ctypes.c_void_p(0x1000), None,
                               ctypes.c_void_p(0x2008), ws, None, ctypes.byref(plan)) == -8
    assert lib.ssd_varlen_plan(ctypes.byref(d), ctypes.c_void_p(0x1000), None,
                               ctypes.c_void_p(0x2000), ws - 1, None, ctypes.byref(plan)) == -8
    assert lib.ssd_varlen_plan(ctypes.byref(d), ctypes.c_void_p(0x1002), None,
                               ctypes.c_void_p(0x2000), ws, None, ctypes.byref(plan)) == -7


def test_forward_rejects_unplanned_and_bad_pointers(lib):
    plan = m.ssd_plan()
    inp = m.ssd_inputs()
    out = m.ssd_outputs()
    assert lib.ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(inp), ctypes.byref(out), None) == -9
    # A plan-shaped struct with the right magic but NULL tensors fails the NULL check.
    plan.dims = _dims()
    plan.magic = 0x5353445641524C31
    plan.workspace = 0x10000
    plan.workspace_bytes = 1 << 30
    plan.seg_len = 2048
    assert lib.ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(inp), ctypes.byref(out), None) == -1
    good = 0x100000
    inp = m.ssd_inputs(good, good, good, good, good, good, None, None, None, None)
    out = m.ssd_outputs(good, None, None, None, None)
    bad = m.ssd_inputs(good + 8, good, good, good, good, good, None, None, None, None)
    assert lib.ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(bad), ctypes.byref(out), None) == -7
    # Using slots without a pool.
    withslots = m.ssd_inputs(good, good, good, good, good, good, None, None, good, None)
    assert lib.ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(withslots), ctypes.byref(out), None) == -1
    # A block table without block_size.
    plan.dims = _dims(block_size=0)
    bt_out = m.ssd_outputs(good, None, None, None, good)
    pool_in = m.ssd_inputs(good, good, good, good, good, good, None, None, None, good)
    assert lib.ssd_varlen_forward(ctypes.byref(plan), ctypes.byref(pool_in), ctypes.byref(bt_out), None) == -5


def test_strerror_names_the_power_of_two_rule(lib):
    assert "power of 2" in m.ssd_varlen_strerror(-3)
    assert m.ssd_varlen_strerror(0) == "ok"


@pytest.mark.parametrize("seed", range(5))
def test_count_chunks_matches_checkpoint_definition(lib, seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 20))
    lens = rng.integers(0, 700, R)
    ncomp = rng.integers(0, 1000, R)
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    for Q in (16, 32, 64, 128, 256):
        _, first = checkpoints.checkpoint_records(lens, ncomp, Q)
        assert m.ssd_varlen_count_chunks(cu, ncomp, Q) == first[-1]
        _, first0 = checkpoints.checkpoint_records(lens, None, Q)
        assert m.ssd_varlen_count_chunks(cu, None, Q) == first0[-1]


# ---- decode step: host validation (no launch is reached) -------------------
_FAKE = 0x100000  # an aligned address the host code never dereferences


def _decode_io(**kw):
    f = ctypes.c_void_p(_FAKE)
    fields = dict(x=f, dt=f, dt_bias=f, A=f, B=f, C=f, D=None, z=None, state_pool=f,
                  read_slots=f, write_slots=None, y=f, device_err=f)
    fields.update(kw)
    return m.ssd_decode_io(*[fields[n] for n, _ in m.ssd_decode_io._fields_])


@pytest.mark.parametrize("kw,code", [
    (dict(R=0), -2), (dict(num_slots=0), -2), (dict(G=3), -4), (dict(dtype=9), -6),
    (dict(N=96), -11), (dict(N=8), -11), (dict(N=512), -11), (dict(P=256, N=128), -11),
])
def test_decode_rejects_bad_dims(lib, kw, code):
    base = dict(T=8, R=2, H=4, P=64, N=128, G=1, chunk_size=0, dtype=m.DTYPE_BF16, num_slots=4)
    base.update(kw)
    d = m.make_dims(**base)
    io = _decode_io()
    assert lib.ssd_varlen_decode(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == code


@pytest.mark.parametrize("field,value,code", [
    ("x", None, -1), ("state_pool", None, -1), ("read_slots", None, -1), ("device_err", None, -1),
    ("y", None, -1), ("x", ctypes.c_void_p(_FAKE + 4), -7), ("read_slots", ctypes.c_void_p(_FAKE + 2), -7),
])
def test_decode_rejects_bad_pointers(lib, field, value, code):
    d = m.make_dims(8, 2, 4, 64, 128, 1, 0, m.DTYPE_BF16, num_slots=4)
    io = _decode_io(**{field: value})
    assert lib.ssd_varlen_decode(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == code
    assert lib.ssd_varlen_decode(ctypes.byref(d), None, ctypes.byref(io), None) == -1


# ---- varlen causal conv1d: host validation ----------------------------------
def _conv_io(**kw):
    f = ctypes.c_void_p(_FAKE)
    fields = dict(x=f, weight=f, bias=None, conv_pool=f, read_slots=f, write_slots=f, y=f, device_err=f)
    fields.update(kw)
    return m.ssd_conv_io(*[fields[n] for n, _ in m.ssd_conv_io._fields_])


def test_conv_struct_sizes():
    assert ctypes.sizeof(m.ssd_conv_dims) == 32
    assert ctypes.sizeof(m.ssd_conv_io) == 8 * 8


@pytest.mark.parametrize("kw,code", [
    (dict(R=0), -2), (dict(D=0), -2), (dict(T=-1), -2), (dict(dtype=4), -6), (dict(W=1), -11),
    (dict(W=5), -11), (dict(D=12), -11),
])
def test_conv_rejects_bad_dims(lib, kw, code):
    base = dict(T=8, R=2, D=64, W=4, dtype=m.DTYPE_BF16, num_slots=4, silu=1)
    base.update(kw)
    d = m.ssd_conv_dims(*[base[n] for n, _ in m.ssd_conv_dims._fields_])
    assert lib.ssd_varlen_conv1d(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(_conv_io()), None) == code


@pytest.mark.parametrize("field,value,code", [
    ("x", None, -1), ("weight", None, -1), ("y", None, -1), ("device_err", None, -1), ("conv_pool", None, -1),
    ("x", ctypes.c_void_p(_FAKE + 8), -7), ("weight", ctypes.c_void_p(_FAKE + 2), -7),
])
def test_conv_rejects_bad_pointers(lib, field, value, code):
    d = m.ssd_conv_dims(8, 2, 64, 4, m.DTYPE_BF16, 4, 1)
    io = _conv_io(**{field: value})
    assert lib.ssd_varlen_conv1d(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == code


# ---- gated delta rule prefill: host validation -------------------------------
def _gdn_io(**kw):
    f = ctypes.c_void_p(_FAKE)
    fields = dict(q=f, k=f, v=f, g=f, beta=f, num_computed=None, state_pool=f, init_slots=f, final_slots=f,
                  block_table=None, o=f, final_states=f, chunk_states=None, device_err=f)
    fields.update(kw)
    return m.ssd_gdn_io(*[fields[n] for n, _ in m.ssd_gdn_io._fields_])


def _gdn_dims(**kw):
    base = dict(T=64, R=2, Hk=2, Hv=4, K=128, V=64, chunk_size=64, block_size=0, block_table_width=0,
                dtype=m.DTYPE_BF16, num_slots=8, l2norm=1, scale=0.0)
    base.update(kw)
    return m.ssd_gdn_dims(*[base[n] for n, _ in m.ssd_gdn_dims._fields_])


def test_gdn_struct_sizes():
    assert ctypes.sizeof(m.ssd_gdn_dims) == 8 + 12 * 4
    assert ctypes.sizeof(m.ssd_gdn_io) == 14 * 8


@pytest.mark.parametrize("kw,code", [
    (dict(R=0), -2), (dict(T=-1), -2), (dict(Hk=0), -2), (dict(num_slots=-1), -2), (dict(Hv=6, Hk=4), -4),
    (dict(dtype=7), -6), (dict(dtype=m.DTYPE_F32), -11), (dict(K=64), -11), (dict(V=48), -11), (dict(V=512), -11),
    (dict(chunk_size=128), -11),
])
def test_gdn_rejects_bad_dims(lib, kw, code):
    d = _gdn_dims(**kw)
    assert lib.ssd_varlen_gdn_forward(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(_gdn_io()), None) == code


@pytest.mark.parametrize("field,value,code", [
    ("q", None, -1), ("k", None, -1), ("v", None, -1), ("g", None, -1), ("beta", None, -1), ("o", None, -1),
    ("device_err", None, -1), ("state_pool", None, -1),
    ("q", ctypes.c_void_p(_FAKE + 8), -7), ("final_states", ctypes.c_void_p(_FAKE + 4), -7),
    ("beta", ctypes.c_void_p(_FAKE + 2), -7),
])
def test_gdn_rejects_bad_pointers(lib, field, value, code):
    io = _gdn_io(**{field: value})
    assert lib.ssd_varlen_gdn_forward(ctypes.byref(_gdn_dims()), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == code
    assert lib.ssd_varlen_gdn_forward(ctypes.byref(_gdn_dims()), None, ctypes.byref(io), None) == -1


def test_gdn_block_table_needs_a_chunk_multiple_block_size(lib):
    io = _gdn_io(block_table=ctypes.c_void_p(_FAKE))
    for bs in (0, 96):
        d = _gdn_dims(block_size=bs, block_table_width=4)
        assert lib.ssd_varlen_gdn_forward(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == -5


def test_gdn_empty_batch_accepts_null_token_buffers(lib):
    # T = 0: q, k, v, g, beta and o may be NULL; validation passes and the call
    # goes on to the launch (which reports SSD_ERR_CUDA on a host without a GPU).
    d = _gdn_dims(T=0)
    io = _gdn_io(q=None, k=None, v=None, g=None, beta=None, o=None)
    rc = lib.ssd_varlen_gdn_forward(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None)
    assert rc not in (-1, -2, -7)
    io = _gdn_io(device_err=None)
    assert lib.ssd_varlen_gdn_forward(ctypes.byref(d), ctypes.c_void_p(_FAKE), ctypes.byref(io), None) == -1


def test_check_slots_host_validation(lib):
    d = m.make_dims(8, 2, 4, 64, 128, 1, 64, m.DTYPE_BF16, num_slots=4)
    f = ctypes.c_void_p(_FAKE)
    assert lib.ssd_varlen_check_slots(ctypes.byref(d), f, f, None, None, None) == -1
    assert lib.ssd_varlen_check_slots(None, f, f, None, f, None) == -1
    bad = m.make_dims(8, 0, 4, 64, 128, 1, 64, m.DTYPE_BF16, num_slots=4)
    assert lib.ssd_varlen_check_slots(ctypes.byref(bad), f, f, None, f, None) == -2
