"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import selective_state_space_154_b300 as ssm
from selective_state_space_154_b300 import build as ssm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ssm_build.build()
    return ssm.load_library()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_header_declares_the_calls():
    names = declared_functions()
    for required in ("ssm_scan_fwd", "ssm_step", "ssm_scan_workspace_bytes", "ssm_scan_check",
                     "ssm_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["SSM_OK", "SSM_ERR_INVALID_ARG", "SSM_ERR_UNSUPPORTED", "SSM_ERR_ALIGNMENT",
                                 "SSM_ERR_WORKSPACE", "SSM_ERR_CUDA", "SSM_ERR_TIMEOUT"]):
        assert ssm.ssm_status_string(code) == name
    assert ssm.ssm_status_string(99) == "SSM_ERR_UNKNOWN"


def _dims(batch=2, d_inner=8, d_state=16, seqlen=64, act=ssm.SSM_DTYPE_BF16):
    return ssm.ssm_dims(batch, d_inner, d_state, seqlen, act, 0)


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced (validation fails first)


def _scan(lib, dims, ptrs=None, ws=None, ws_bytes=0):
    p = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, out=FAKE, fs=None)
    p.update(ptrs or {})
    args = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("u", "delta", "A", "B", "C", "D", "z", "bias", "out", "fs")]
    return lib.ssm_scan_fwd(*args, ctypes.byref(dims), ws, ws_bytes, None)


def _step(lib, dims, ptrs=None):
    p = dict(state=FAKE, x=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, out=FAKE)
    p.update(ptrs or {})
    args = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("state", "x", "delta", "A", "B", "C", "D", "z", "bias", "out")]
    return lib.ssm_step(*args, ctypes.byref(dims), None)


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, ssm.SSM_ERR_INVALID_ARG), ("d_inner", -1, ssm.SSM_ERR_INVALID_ARG),
    ("d_state", 0, ssm.SSM_ERR_INVALID_ARG), ("seqlen", 0, ssm.SSM_ERR_INVALID_ARG),
    ("act", 7, ssm.SSM_ERR_INVALID_ARG), ("d_state", 65, ssm.SSM_ERR_UNSUPPORTED),
    ("seqlen", 1 << 61, ssm.SSM_ERR_UNSUPPORTED),
])
def test_scan_rejects_bad_dims(lib, field, value, status):
    d = _dims()
    setattr(d, field, value)
    assert _scan(lib, d) == status
    assert lib.ssm_scan_workspace_bytes(ctypes.byref(d)) == 0


def test_scan_rejects_null_dims(lib):
    args = [ctypes.c_void_p(FAKE)] * 5 + [None] * 3 + [ctypes.c_void_p(FAKE), None]
    assert lib.ssm_scan_fwd(*args, None, None, 0, None) == ssm.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("missing", ["u", "delta", "A", "B", "C", "out"])
def test_scan_rejects_null_required_pointer(lib, missing):
    assert _scan(lib, _dims(), {missing: None}) == ssm.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["u", "delta", "B", "C", "z", "out"])
def test_scan_rejects_misaligned_activation_pointer(lib, which):
    assert _scan(lib, _dims(), {which: FAKE + 1}) == ssm.SSM_ERR_ALIGNMENT          # bf16: 2-byte
    assert _scan(lib, _dims(act=ssm.SSM_DTYPE_F32), {which: FAKE + 2}) == ssm.SSM_ERR_ALIGNMENT


@pytest.mark.parametrize("which", ["u", "delta", "B", "C", "z", "out"])
def test_scan_accepts_element_aligned_pointers(lib, which):
    """Element alignment is the rule: a bf16 pointer 2 bytes past a 16-byte boundary
    (an fp32 one 4 bytes past) passes validation and reaches the launch, which here,
    with no GPU, fails as a CUDA error rather than as an alignment error."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the fake pointers would be dereferenced by a real launch")
    for act, off in ((ssm.SSM_DTYPE_BF16, 2), (ssm.SSM_DTYPE_F32, 4)):
        st = _scan(lib, _dims(act=act), {which: FAKE + off})
        assert st == ssm.SSM_ERR_CUDA, ssm.ssm_status_string(st)


def test_noalloc_scratch_size_matches_the_header(lib):
    text = open(os.path.join(ROOT, "include", "ssm_scan.h")).read()
    m = re.search(r"#define SSM_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m
    assert lib.ssm_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))
    assert ssm.SSM_NOALLOC_SCRATCH_BYTES == lib.ssm_noalloc_scratch_bytes()


@pytest.mark.parametrize("which", ["A", "D", "bias", "fs"])
def test_scan_rejects_misaligned_fp32_pointer(lib, which):
    assert _scan(lib, _dims(), {which: FAKE + 2}) == ssm.SSM_ERR_ALIGNMENT


@pytest.mark.parametrize("missing", ["state", "x", "delta", "A", "B", "C", "out"])
def test_step_rejects_null_required_pointer(lib, missing):
    assert _step(lib, _dims(), {missing: None}) == ssm.SSM_ERR_INVALID_ARG


def test_step_rejects_bad_dims_and_alignment(lib):
    d = _dims(d_state=100)
    assert _step(lib, d) == ssm.SSM_ERR_UNSUPPORTED
    d = _dims(d_inner=0)
    assert _step(lib, d) == ssm.SSM_ERR_INVALID_ARG
    assert _step(lib, _dims(), {"state": FAKE + 4}) == ssm.SSM_ERR_ALIGNMENT   # state: 16-byte
    assert _step(lib, _dims(), {"A": FAKE + 8}) == ssm.SSM_ERR_ALIGNMENT
    assert _step(lib, _dims(), {"x": FAKE + 1}) == ssm.SSM_ERR_ALIGNMENT


def test_long_sequence_needs_workspace(lib):
    """A long sequence over few rows is split into chunks, which needs workspace;
    without it the call is rejected before any launch."""
    d = _dims(batch=1, d_inner=64, d_state=16, seqlen=1 << 20)
    need = lib.ssm_scan_workspace_bytes(ctypes.byref(d))
    assert need > 0
    assert _scan(lib, d) == ssm.SSM_ERR_WORKSPACE
    assert _scan(lib, d, ws=ctypes.c_void_p(FAKE), ws_bytes=need - 1) == ssm.SSM_ERR_WORKSPACE


def test_short_sequence_needs_no_workspace(lib):
    d = _dims(batch=64, d_inner=4096, d_state=16, seqlen=256)
    assert lib.ssm_scan_workspace_bytes(ctypes.byref(d)) == 0


def test_check_without_workspace_is_ok(lib):
    assert lib.ssm_scan_check(None, 0) == ssm.SSM_OK


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    u = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError):
        ssm.scan_fwd(u, u, torch.zeros(1, 4), torch.zeros(1, 8, 4), torch.zeros(1, 8, 4))


def _scan_from(lib, dims, h0, ptrs=None):
    p = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, out=FAKE, fs=None)
    p.update(ptrs or {})
    a = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("u", "delta", "A", "B", "C", "D", "z", "bias")]
    tail = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("out", "fs")]
    return lib.ssm_scan_fwd_from_state(*a, ctypes.c_void_p(h0) if h0 else None, *tail, ctypes.byref(dims),
                                       None, 0, None)


def test_scan_from_state_validates_the_initial_state(lib):
    assert _scan_from(lib, _dims(), None) == ssm.SSM_ERR_INVALID_ARG       # required
    assert _scan_from(lib, _dims(), FAKE + 2) == ssm.SSM_ERR_ALIGNMENT     # float32: 4-byte aligned
    d = _dims()
    d.seqlen = 0
    assert _scan_from(lib, d, FAKE) == ssm.SSM_ERR_INVALID_ARG             # dims checked as for ssm_scan_fwd
    assert _scan_from(lib, _dims(), FAKE, {"u": None}) == ssm.SSM_ERR_INVALID_ARG


def _conv(lib, dims, width=4, ptrs=None):
    p = dict(x=FAKE, w=FAKE, bias=None, s0=None, out=FAKE, sT=None)
    p.update(ptrs or {})
    a = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("x", "w", "bias", "s0", "out", "sT")]
    return lib.ssm_conv1d_fwd(*a, ctypes.byref(dims), width, None)


def _conv_step(lib, dims, width=4, ptrs=None):
    p = dict(state=FAKE, x=FAKE, w=FAKE, bias=None, out=FAKE)
    p.update(ptrs or {})
    a = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("state", "x", "w", "bias", "out")]
    return lib.ssm_conv1d_step(*a, ctypes.byref(dims), width, None)


@pytest.mark.parametrize("width,status", [(0, ssm.SSM_ERR_INVALID_ARG), (-3, ssm.SSM_ERR_INVALID_ARG),
                                          (9, ssm.SSM_ERR_UNSUPPORTED)])
def test_conv_rejects_bad_width(lib, width, status):
    assert _conv(lib, _dims(), width) == status
    assert _conv_step(lib, _dims(), width) == status


@pytest.mark.parametrize("missing", ["x", "w", "out"])
def test_conv_rejects_null_required_pointer(lib, missing):
    assert _conv(lib, _dims(), ptrs={missing: None}) == ssm.SSM_ERR_INVALID_ARG
    assert _conv_step(lib, _dims(), ptrs={missing: None}) == ssm.SSM_ERR_INVALID_ARG


def test_conv_step_needs_a_state_unless_width_one(lib):
    assert _conv_step(lib, _dims(), 4, {"state": None}) == ssm.SSM_ERR_INVALID_ARG


def test_conv_rejects_misaligned_and_bad_dims(lib):
    assert _conv(lib, _dims(), ptrs={"x": FAKE + 1}) == ssm.SSM_ERR_ALIGNMENT
    assert _conv(lib, _dims(), ptrs={"sT": FAKE + 1}) == ssm.SSM_ERR_ALIGNMENT
    assert _conv(lib, _dims(), ptrs={"w": FAKE + 2}) == ssm.SSM_ERR_ALIGNMENT
    assert _conv_step(lib, _dims(), ptrs={"state": FAKE + 1}) == ssm.SSM_ERR_ALIGNMENT
    d = _dims()
    d.seqlen = 0
    assert _conv(lib, d) == ssm.SSM_ERR_INVALID_ARG
    d = _dims()
    d.act = 5
    assert _conv_step(lib, d) == ssm.SSM_ERR_INVALID_ARG


def _ssd_dims(batch=2, seqlen=300, nheads=4, headdim=64, ngroups=2, d_state=128, act=ssm.SSM_DTYPE_BF16):
    return ssm.ssd_dims(batch, seqlen, nheads, headdim, ngroups, d_state, act, 0)


def _ssd(lib, dims, ptrs=None, ws=FAKE, ws_bytes=1 << 40):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, h0=None, out=FAKE, fs=None)
    p.update(ptrs or {})
    args = [ctypes.c_void_p(p[k]) if p[k] else None
            for k in ("x", "dt", "A", "B", "C", "D", "z", "bias", "h0", "out", "fs")]
    return lib.ssd_scan_fwd(*args, ctypes.byref(dims), ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, ssm.SSM_ERR_INVALID_ARG), ("nheads", 0, ssm.SSM_ERR_INVALID_ARG),
    ("ngroups", 3, ssm.SSM_ERR_INVALID_ARG), ("seqlen", -1, ssm.SSM_ERR_INVALID_ARG),
    ("act", 5, ssm.SSM_ERR_INVALID_ARG), ("act", ssm.SSM_DTYPE_F32, ssm.SSM_ERR_UNSUPPORTED),
    ("headdim", 32, ssm.SSM_ERR_UNSUPPORTED), ("d_state", 64, ssm.SSM_ERR_UNSUPPORTED),
    ("nheads", 1 << 17, ssm.SSM_ERR_UNSUPPORTED),
])
def test_ssd_rejects_bad_dims(lib, field, value, status):
    d = _ssd_dims()
    setattr(d, field, value)
    assert _ssd(lib, d) == status
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(d)) == 0


@pytest.mark.parametrize("missing", ["x", "dt", "A", "B", "C", "out"])
def test_ssd_rejects_null_required_pointer(lib, missing):
    assert _ssd(lib, _ssd_dims(), {missing: None}) == ssm.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("which,offset", [("x", 2), ("z", 8), ("out", 2), ("B", 4), ("C", 2), ("dt", 1),
                                          ("A", 2), ("D", 1), ("bias", 2), ("h0", 2), ("fs", 1)])
def test_ssd_rejects_misaligned_pointer(lib, which, offset):
    assert _ssd(lib, _ssd_dims(), {which: FAKE + offset}) == ssm.SSM_ERR_ALIGNMENT


def test_ssd_workspace_size_and_check(lib):
    d = _ssd_dims()
    need = lib.ssd_scan_workspace_bytes(ctypes.byref(d))
    # 3 chunks of 128 tokens per (batch, head): fp32 chunk states, the two bf16 terms of the
    # incoming states and the chunk decays
    cells = 2 * 4 * 3
    assert need >= 256 + cells * 64 * 128 * (4 + 2 * 2) + cells * 4
    assert _ssd(lib, d, ws_bytes=need - 1) == ssm.SSM_ERR_WORKSPACE
    assert _ssd(lib, d, ws=None, ws_bytes=0) == ssm.SSM_ERR_WORKSPACE
    assert _ssd(lib, d, ws=FAKE + 8, ws_bytes=need) == ssm.SSM_ERR_ALIGNMENT


def _ssd_step(lib, dims, ptrs=None):
    p = dict(state=FAKE, x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, out=FAKE)
    p.update(ptrs or {})
    args = [ctypes.c_void_p(p[k]) if p[k] else None
            for k in ("state", "x", "dt", "A", "B", "C", "D", "z", "bias", "out")]
    return lib.ssd_step(*args, ctypes.byref(dims), None)


@pytest.mark.parametrize("missing", ["state", "x", "dt", "A", "B", "C", "out"])
def test_ssd_step_rejects_null_required_pointer(lib, missing):
    assert _ssd_step(lib, _ssd_dims(), {missing: None}) == ssm.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("which,offset", [("state", 4), ("B", 8), ("C", 2), ("x", 1), ("out", 1), ("A", 2)])
def test_ssd_step_rejects_misaligned_pointer(lib, which, offset):
    assert _ssd_step(lib, _ssd_dims(), {which: FAKE + offset}) == ssm.SSM_ERR_ALIGNMENT


def test_ssd_step_rejects_unsupported_dims(lib):
    assert _ssd_step(lib, _ssd_dims(d_state=64)) == ssm.SSM_ERR_UNSUPPORTED
    assert _ssd_step(lib, _ssd_dims(ngroups=3)) == ssm.SSM_ERR_INVALID_ARG


def _host_scan(lib, dims, piece, staging=None, staging_bytes=0, ptrs=None):
    p = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, h0=None, out=FAKE, fs=None)
    p.update(ptrs or {})
    a = [ctypes.c_void_p(p[k]) if p[k] else None for k in ("u", "delta", "A", "B", "C", "D", "z", "bias", "h0",
                                                          "out", "fs")]
    return lib.ssm_scan_fwd_host(*a, ctypes.byref(dims), piece, staging, staging_bytes, None, None, None)


def test_host_scan_validates_before_any_copy(lib):
    d = _dims(batch=1, d_inner=64, d_state=16, seqlen=10000)
    need = lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), 4096)
    assert need > 0
    # a larger piece needs more staging; pieces longer than the sequence count as the sequence
    assert lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), 8192) > need
    assert lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), 1 << 30) == \
        lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), 10000)
    assert lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), 0) == 0
    assert _host_scan(lib, d, 0) == ssm.SSM_ERR_INVALID_ARG
    assert _host_scan(lib, d, 4096) == ssm.SSM_ERR_WORKSPACE
    assert _host_scan(lib, d, 4096, ctypes.c_void_p(FAKE), need - 1) == ssm.SSM_ERR_WORKSPACE
    assert _host_scan(lib, d, 4096, ctypes.c_void_p(FAKE + 16), need) == ssm.SSM_ERR_ALIGNMENT
    assert _host_scan(lib, d, 4096, ctypes.c_void_p(FAKE), need, {"out": None}) == ssm.SSM_ERR_INVALID_ARG
    bad = _dims(d_state=65)
    assert _host_scan(lib, bad, 16, ctypes.c_void_p(FAKE), 1 << 30) == ssm.SSM_ERR_UNSUPPORTED


def test_ssd_walking_form_workspace(lib, hooks):
    """batch · nheads ≥ 64 selects the form where one CTA walks each (batch, head): with
    every unit walked whole its workspace is the 256 bytes of error words; units cut into
    segments add a flag, a decay and a 64 × 128 fp32 state per segment; the chunk-parallel
    form (forced, or below the threshold) needs the chunk states besides."""
    many = _ssd_dims(batch=2, nheads=40, ngroups=4)  # 80 units, 3 chunks: each walked whole
    few = _ssd_dims()
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(many)) == 256
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(few)) > 256
    assert _ssd(lib, many, ws_bytes=255) == ssm.SSM_ERR_WORKSPACE
    hooks.set("SSM_FORCE_KERNEL", "ssd_chunks")
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(many)) > 256
    hooks.set("SSM_FORCE_KERNEL", "ssd_walk")
    hooks.set("SSM_SSD_SPLIT", 3)  # 8 units × 3 segments
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(few)) == 256 + 256 + 256 + 24 * 64 * 128 * 4  # 25 words fit
