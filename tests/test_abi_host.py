"""Host-side checks of the C ABI, no GPU needed: the library builds and loads, exports
every entry point include/ssmscan.h declares, and rejects bad arguments before it
launches anything (so these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

from selective_scan_mamba_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ssmscan.h")).read()
    return sorted(set(re.findall(
        r"^\s*(?:ssm_status|size_t|int|unsigned int|const char\*)\s+(\w+)\s*\(", text, re.M)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("ssm_scan_fwd", "ssd_chunk_scan_fwd", "ssm_state_update"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(_lib.SYMBOLS) <= set(declared_functions())


def test_abi_version(lib):
    assert lib.ssm_abi_version() == 2 == _lib.ABI_VERSION



FAKE = 0x7F0000000000  # a 16-byte aligned address; never dereferenced by these calls


def fake(i):
    """The i-th of a set of far-apart aligned fake addresses (distinct tensors, so that the
    overlap checks pass); never dereferenced by these calls."""
    return FAKE + (i << 36)


def set_fakes(p, fields):
    for i, f in enumerate(fields):
        setattr(p, f, fake(i + 1))


def scan_params(**kw):
    p = _lib.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen, p.ngroups = 2, 32, 16, 64, 1
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    set_fakes(p, ("x", "delta", "A", "B", "C", "y"))
    p.delta_softplus = 1
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, _lib.SSM_ERR_INVALID_ARG),
    ("dim", -1, _lib.SSM_ERR_INVALID_ARG),
    ("seqlen", -5, _lib.SSM_ERR_INVALID_ARG),
    ("ngroups", 3, _lib.SSM_ERR_INVALID_ARG),   # does not divide dim
    ("in_dtype", 7, _lib.SSM_ERR_INVALID_ARG),
    ("disc", 9, _lib.SSM_ERR_INVALID_ARG),
    ("dstate", 300, _lib.SSM_ERR_UNSUPPORTED),
    ("x", None, _lib.SSM_ERR_INVALID_ARG),
    ("y", FAKE + 8, _lib.SSM_ERR_INVALID_ARG),  # misaligned
    ("A", None, _lib.SSM_ERR_INVALID_ARG),
    ("h0", FAKE + 4, _lib.SSM_ERR_INVALID_ARG),
])
def test_scan_rejects_bad_arguments(lib, field, value, status):
    p = scan_params(**{field: value})
    rc = lib.ssm_scan_fwd(ctypes.byref(p), None)
    assert rc == status
    assert lib.ssm_last_error().decode()
    o = _lib.ScanOpts()
    assert lib.ssm_scan_fwd_ex(ctypes.byref(p), ctypes.byref(o), fake(30), 1 << 30, None) == status


def test_scan_null_params(lib):
    assert lib.ssm_scan_fwd(None, None) == _lib.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_fwd_ex(None, None, None, 0, None) == _lib.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_workspace_size(None, None) == 0


@pytest.mark.parametrize("field,value", [("kernel", 9), ("threads_per_channel", 3),
                                         ("max_segments", -1), ("fault_test", 2)])
def test_scan_rejects_bad_options(lib, field, value):
    o = _lib.ScanOpts()
    setattr(o, field, value)
    assert lib.ssm_scan_fwd_ex(ctypes.byref(scan_params()), ctypes.byref(o), None, 0, None) == \
        _lib.SSM_ERR_INVALID_ARG
    assert field in lib.ssm_last_error().decode()
    assert lib.ssm_scan_workspace_size(ctypes.byref(scan_params()), ctypes.byref(o)) == 0


def test_scan_kernel_that_cannot_run_the_problem_is_unsupported(lib):
    """Naming a kernel that does not take the problem (the TMEM kernel needs bf16 inputs
    and dstate 16) is refused on the host."""
    o = _lib.ScanOpts()
    o.kernel = _lib.SSM_SCAN_KERNEL_TMEM
    p = scan_params(dstate=8)
    assert lib.ssm_scan_fwd_ex(ctypes.byref(p), ctypes.byref(o), None, 0, None) == \
        _lib.SSM_ERR_UNSUPPORTED
    assert "TMEM" in lib.ssm_last_error().decode()


@pytest.mark.parametrize("out,inp", [("y", "x"), ("y", "B"), ("h_final", "h0"), ("y", "h_final")])
def test_scan_refuses_overlapping_outputs(lib, out, inp):
    """An output that overlaps an input (or another output) is refused before any launch."""
    p = scan_params(h0=fake(20), h_final=fake(21))
    setattr(p, out, getattr(p, inp) + 64)  # inside the other tensor
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == _lib.SSM_ERR_INVALID_ARG
    assert "overlaps" in lib.ssm_last_error().decode()


@pytest.mark.gpu
def test_workspace_overlapping_an_input_is_refused(lib):
    """The time-split plan's workspace must not overlap the tensors (one batch row, few
    channels, long sequence: the automatic plan splits it)."""
    p = scan_params(batch=1, dim=256, seqlen=4096)
    o = _lib.ScanOpts()
    need = lib.ssm_scan_workspace_size(ctypes.byref(p), ctypes.byref(o))
    assert need > 0
    assert lib.ssm_scan_fwd_ex(ctypes.byref(p), ctypes.byref(o), p.x, need, None) == \
        _lib.SSM_ERR_INVALID_ARG


def ssd_params(**kw):
    p = _lib.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = 2, 256, 4, 64, 128, 1, 64
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    set_fakes(p, ("x", "dt", "A", "B", "C", "y"))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,status", [
    ("chunk_size", 100, _lib.SSM_ERR_UNSUPPORTED),
    ("headdim", 48, _lib.SSM_ERR_UNSUPPORTED),
    ("dstate", 16, _lib.SSM_ERR_UNSUPPORTED),
    ("ngroups", 3, _lib.SSM_ERR_INVALID_ARG),
    ("nheads", 0, _lib.SSM_ERR_INVALID_ARG),
    ("B", None, _lib.SSM_ERR_INVALID_ARG),
    ("dt", FAKE + 2, _lib.SSM_ERR_INVALID_ARG),
])
def test_ssd_rejects_bad_arguments(lib, field, value, status):
    p = ssd_params(**{field: value})
    need = lib.ssd_chunk_scan_workspace_size(ctypes.byref(p))
    rc = lib.ssd_chunk_scan_fwd(ctypes.byref(p), fake(30), max(need, 1 << 30), None)
    assert rc == status


def test_ssd_refuses_overlaps(lib):
    p = ssd_params()
    need = lib.ssd_chunk_scan_workspace_size(ctypes.byref(p))
    p.y = p.x
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), fake(30), need, None) == _lib.SSM_ERR_INVALID_ARG
    assert "overlaps" in lib.ssm_last_error().decode()
    p = ssd_params()
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), p.C, need, None) == _lib.SSM_ERR_INVALID_ARG
    assert "workspace" in lib.ssm_last_error().decode()


def test_ssd_workspace_size_and_shortfall(lib):
    p = ssd_params(headdim=32)  # CUDA-core path: one fp32 state per chunk
    need = lib.ssd_chunk_scan_workspace_size(ctypes.byref(p))
    nch = 256 // 64
    assert need >= 2 * 4 * nch * 32 * 128 * 4
    rc = lib.ssd_chunk_scan_fwd(ctypes.byref(p), fake(30), need - 1, None)
    assert rc == _lib.SSM_ERR_INVALID_ARG
    assert "workspace" in lib.ssm_last_error().decode()
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(ssd_params(chunk_size=7))) == 0


def step_params(**kw):
    p = _lib.StepParams()
    p.batch, p.nheads, p.headdim, p.dstate, p.ngroups = 4, 8, 16, 64, 1
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    set_fakes(p, ("state", "x", "dt", "A", "B", "C", "y"))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_step_refuses_y_inside_the_state(lib):
    """The state is updated in place by design, but y may not overlap it or an input."""
    p = step_params()
    p.y = p.state + 256
    assert lib.ssm_state_update(ctypes.byref(p), None) == _lib.SSM_ERR_INVALID_ARG
    assert "overlaps" in lib.ssm_last_error().decode()
    p = step_params()
    p.state = p.B
    assert lib.ssm_state_update(ctypes.byref(p), None) == _lib.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("ntokens", [0, -1, 257])
def test_step_tokens_rejects_bad_count(lib, ntokens):
    p = step_params()
    assert lib.ssm_state_update_tokens(ctypes.byref(p), ntokens, None) == _lib.SSM_ERR_INVALID_ARG
    assert "ntokens" in lib.ssm_last_error().decode()


@pytest.mark.parametrize("field,value,status", [
    ("state", None, _lib.SSM_ERR_INVALID_ARG),
    ("a_per_state", 2, _lib.SSM_ERR_INVALID_ARG),
    ("ngroups", 3, _lib.SSM_ERR_INVALID_ARG),
    ("headdim", 0, _lib.SSM_ERR_INVALID_ARG),
    ("z", FAKE + 1, _lib.SSM_ERR_INVALID_ARG),
])
def test_step_rejects_bad_arguments(lib, field, value, status):
    p = step_params(**{field: value})
    assert lib.ssm_state_update(ctypes.byref(p), None) == status


def test_injected_launch_fault_reports_cuda_error(lib, monkeypatch):
    """The host-side fault hook turns a valid call into SSM_ERR_CUDA before any CUDA call."""
    monkeypatch.setenv("SSM_FAULT_INJECT", "launch")
    assert lib.ssm_state_update(ctypes.byref(step_params()), None) == _lib.SSM_ERR_CUDA
    assert "injected" in lib.ssm_last_error().decode()
    assert lib.ssm_scan_fwd(ctypes.byref(scan_params()), None) == _lib.SSM_ERR_CUDA
    p = ssd_params()
    need = lib.ssd_chunk_scan_workspace_size(ctypes.byref(p))
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), fake(30), need, None) == _lib.SSM_ERR_CUDA


def test_python_binding_refuses_cpu_tensors():
    import torch
    import selective_scan_mamba_gb300 as ssm
    x = torch.zeros(1, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        ssm.ssm_scan_fwd(x, x, torch.zeros(4, 16), torch.zeros(1, 16, 8, dtype=torch.bfloat16),
                         torch.zeros(1, 16, 8, dtype=torch.bfloat16))


def test_size_ceilings_refuse_before_any_launch(lib):
    """Problems past the index ranges the kernels use are refused, not wrapped."""
    p = ssd_params(batch=4, seqlen=2**31 - 1)
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), fake(30), 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG
    assert "too large" in lib.ssm_last_error().decode()
    p = step_params(batch=2**28)  # 2^41 state elements
    assert lib.ssm_state_update(ctypes.byref(p), None) == _lib.SSM_ERR_INVALID_ARG
    assert "too large" in lib.ssm_last_error().decode()
    p = step_params(batch=2**26)  # B/C rows of 2^32 elements
    assert lib.ssm_state_update(ctypes.byref(p), None) == _lib.SSM_ERR_UNSUPPORTED
    assert "too large" in lib.ssm_last_error().decode()


# ctypes mirrors of the C parameter structs, by the header's typedef names
C_STRUCTS = {
    "ssm_scan_params": _lib.ScanParams,
    "ssm_scan_bwd_params": _lib.ScanBwdParams,
    "ssm_mamba3_params": _lib.Mamba3Params,
    "ssm_s4d_params": _lib.S4dParams,
    "ssd_params": _lib.SsdParams,
    "ssd_bwd_params": _lib.SsdBwdParams,
    "ssm_step_params": _lib.StepParams,
    "ssm_scan_opts": _lib.ScanOpts,
}


ENUM_CONSTANTS = ("SSM_OK", "SSM_ERR_INVALID_ARG", "SSM_ERR_UNSUPPORTED", "SSM_ERR_CUDA",
                  "SSM_ERR_TIMEOUT", "SSM_F32", "SSM_BF16", "SSM_DISC_EXP_EULER", "SSM_DISC_ZOH",
                  "SSM_SCAN_KERNEL_AUTO", "SSM_SCAN_KERNEL_TMEM", "SSM_SCAN_KERNEL_TMA",
                  "SSM_SCAN_KERNEL_TILED", "SSM_SCAN_KERNEL_GENERIC")


def test_ctypes_structs_match_the_header_layout(tmp_path):
    """Every field offset and every struct size of the Python binding's ctypes mirrors,
    and every enum constant it uses, equals what a C compiler makes of include/ssmscan.h,
    so no argument lands in another field's slot."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ssmscan.h"', 'int main(void) {']
    for cname, cls in C_STRUCTS.items():
        lines.append(f'    printf("{cname} . %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'    printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    for const in ENUM_CONSTANTS:
        lines.append(f'    printf("enum {const} %d\\n", (int){const});')
    lines += ['    return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    seen = 0
    for line in out.splitlines():
        cname, fname, value = line.split()
        if cname == "enum":
            assert int(value) == getattr(_lib, fname), f"{fname}: C says {value}"
            seen += 1
            continue
        cls = C_STRUCTS[cname]
        want = ctypes.sizeof(cls) if fname == "." else getattr(cls, fname).offset
        assert int(value) == want, f"{cname}.{fname}: C says {value}, ctypes says {want}"
        seen += 1
    assert seen == sum(len(c._fields_) + 1 for c in C_STRUCTS.values()) + len(ENUM_CONSTANTS)


def _header_prototypes():
    """(return type, name, [parameter types]) of every function include/ssmscan.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "ssmscan.h")).read(),
                  flags=re.S)
    out = []
    for ret, name, args in re.findall(
            r"^\s*(ssm_status|size_t|int|const char\s*\*|unsigned int)\s+(\w+)\s*\(([^)]*)\)\s*;",
            text, re.M | re.S):
        params = [] if args.strip() == "void" else [
            " ".join(a.split()).rsplit(" ", 1)[0] if not a.strip().endswith("*") else a.strip()
            for a in args.split(",")]
        out.append((" ".join(ret.split()), name, params))
    return out


def _ctype_of(c_type):
    """The ctypes type the binding must declare for a C parameter or return type."""
    t = c_type.replace("const ", "").replace(" *", "*").strip()
    if t.endswith("_params*") or t.endswith("_opts*"):
        return ctypes.POINTER(C_STRUCTS[t[:-1]])
    return {"void*": ctypes.c_void_p, "float*": ctypes.c_void_p, "size_t": ctypes.c_size_t,
            "int": ctypes.c_int, "ssm_status": ctypes.c_int, "char*": ctypes.c_char_p,
            "unsigned int": ctypes.c_uint}[t]


def test_ctypes_signatures_match_the_header(lib):
    """Every function the loader declares has the header's parameter count, parameter
    types and return type; every symbol the binding calls is declared."""
    protos = _header_prototypes()
    assert {n for _, n, _ in protos} >= set(_lib.SYMBOLS) | {"ssm_wait_timeouts"}
    checked = 0
    for ret, name, params in protos:
        fn = getattr(lib, name)
        if fn.argtypes is None:  # not used by the binding (declared by its own test)
            assert name not in _lib.SYMBOLS, name
            continue
        want = [_ctype_of(p) for p in params]
        assert list(fn.argtypes) == want, f"{name}: argtypes {fn.argtypes} != header {params}"
        assert fn.restype == _ctype_of(ret), f"{name}: restype {fn.restype} != header {ret}"
        checked += 1
    assert checked >= len(_lib.SYMBOLS)


def _tensor_on_cuda1(shape):
    """A CPU tensor that reports itself as living on cuda:1, to reach the binding's
    device check without a GPU."""
    import torch

    class OnCuda1(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        @property
        def device(self):
            return torch.device("cuda", 1)

    return torch.Tensor._make_subclass(OnCuda1, torch.zeros(shape))


def test_python_binding_refuses_tensor_of_another_device(monkeypatch):
    import torch
    import selective_scan_mamba_gb300 as ssm
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="current device"):
        ssm._ptr(_tensor_on_cuda1((4,)), "x")


def test_python_binding_refuses_stream_of_another_device(monkeypatch):
    import torch
    import selective_scan_mamba_gb300 as ssm

    class Stream1:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="current device"):
        ssm._stream(Stream1())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    assert ssm._stream(Stream1()).value in (None, 0)


def scan_bwd_params(**kw):
    p = _lib.ScanBwdParams()
    p.fwd = scan_params()
    for i, f in enumerate(("dy", "dx", "ddelta", "dA", "dB", "dC")):
        setattr(p, f, fake(10 + i))
    for k, v in kw.items():
        if k.startswith("fwd_"):
            setattr(p.fwd, k[4:], v)
        else:
            setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    ({"fwd_disc": _lib.SSM_DISC_ZOH}, _lib.SSM_ERR_UNSUPPORTED),
    ({"fwd_dstate": 8}, _lib.SSM_ERR_UNSUPPORTED),
    ({"fwd_dstate": 24}, _lib.SSM_ERR_UNSUPPORTED),
    ({"dA": None}, _lib.SSM_ERR_INVALID_ARG),
    ({"dy": None}, _lib.SSM_ERR_INVALID_ARG),
    ({"dB": FAKE + 4}, _lib.SSM_ERR_INVALID_ARG),
    ({"fwd_z": fake(20)}, _lib.SSM_ERR_INVALID_ARG),            # z given, dz missing
    ({"dD_skip": fake(20)}, _lib.SSM_ERR_INVALID_ARG),          # dD given, D missing
    ({"fwd_delta_bias": fake(20)}, _lib.SSM_ERR_INVALID_ARG),   # bias given, dbias missing
    ({"dx": fake(1)}, _lib.SSM_ERR_INVALID_ARG),                # dx is x
    ({"fwd_ngroups": 3}, _lib.SSM_ERR_INVALID_ARG),
])
def test_scan_bwd_rejects_bad_arguments(lib, kw, status):
    p = scan_bwd_params(**kw)
    assert lib.ssm_scan_bwd(ctypes.byref(p), fake(30), 1 << 40, None) == status
    assert lib.ssm_last_error()


def bwd_workspace_bytes(rows, N, L, in_bytes=2, dy_bytes=2):
    """The backward's scratch: coarse checkpoints (one per block of K 16-step chunks:
    K = 1 while N floats per chunk fit in the bytes of x and dy per 16 steps, else
    ceil(sqrt(chunks))), one block's fine checkpoints when K > 1, per-row dA, dD, dbias
    sums; each part rounded up to 256 bytes."""
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    nch = -(-L // 16)
    kb = 1
    if nch * N * 4 > L * (in_bytes + dy_bytes):
        while kb * kb < nch:
            kb += 1
    nblk = -(-nch // kb)
    fine = r256(rows * kb * N * 4) if kb > 1 else 0
    return r256(rows * nblk * N * 4) + fine + r256(rows * N * 4) + 2 * r256(rows * 4)


def test_scan_bwd_workspace_size_and_shortfall(lib):
    p = scan_bwd_params()
    need = lib.ssm_scan_bwd_workspace_size(ctypes.byref(p))
    assert need == bwd_workspace_bytes(2 * 32, 16, 64)
    assert lib.ssm_scan_bwd(ctypes.byref(p), fake(30), need - 1, None) == _lib.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(scan_bwd_params(fwd_dstate=8))) == 0
    assert lib.ssm_scan_bwd_workspace_size(None) == 0


def mamba3_params(**kw):
    p = _lib.Mamba3Params()
    p.batch, p.dim, p.dstate, p.seqlen, p.ngroups = 2, 32, 16, 64, 1
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    set_fakes(p, ("x", "delta", "A_re", "A_im", "lam", "B", "C", "y"))
    p.delta_softplus = 1
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,status", [
    ("dstate", 12, _lib.SSM_ERR_UNSUPPORTED),
    ("dstate", 128, _lib.SSM_ERR_UNSUPPORTED),
    ("A_im", None, _lib.SSM_ERR_INVALID_ARG),
    ("lam", None, _lib.SSM_ERR_INVALID_ARG),
    ("lam", FAKE + 2, _lib.SSM_ERR_INVALID_ARG),
    ("ngroups", 5, _lib.SSM_ERR_INVALID_ARG),
    ("batch", 0, _lib.SSM_ERR_INVALID_ARG),
])
def test_mamba3_rejects_bad_arguments(lib, field, value, status):
    p = mamba3_params(**{field: value})
    assert lib.ssm_mamba3_scan_fwd(ctypes.byref(p), fake(30), 1 << 40, None) == status
    assert lib.ssm_last_error()


@pytest.mark.parametrize("field,value,status", [
    ("dstate", 6, _lib.SSM_ERR_UNSUPPORTED),
    ("log_dt", None, _lib.SSM_ERR_INVALID_ARG),
    ("C", FAKE + 8, _lib.SSM_ERR_INVALID_ARG),
    ("u", None, _lib.SSM_ERR_INVALID_ARG),
    ("batch", 0, _lib.SSM_ERR_INVALID_ARG),
])
def test_s4d_rejects_bad_arguments(lib, field, value, status):
    p = _lib.S4dParams()
    p.batch, p.dim, p.dstate, p.seqlen = 2, 16, 32, 64
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    set_fakes(p, ("u", "log_dt", "A", "B", "C", "y"))
    setattr(p, field, value)
    assert lib.ssm_s4d_scan_fwd(ctypes.byref(p), fake(30), 1 << 40, None) == status
    if field in ("dstate", "log_dt", "C"):
        assert lib.ssm_s4d_kernel(ctypes.byref(p), fake(31), 16, None) == status


def ssd_bwd_params(**kw):
    p = _lib.SsdBwdParams()
    f = p.fwd
    f.batch, f.seqlen, f.nheads, f.headdim, f.dstate, f.ngroups, f.chunk_size = 2, 64, 4, 64, 128, 1, 64
    f.in_dtype = f.out_dtype = _lib.SSM_BF16
    set_fakes(f, ("x", "dt", "A", "B", "C"))
    f.dt_softplus = 1
    for i, n in enumerate(("dy", "dx", "ddt", "dA", "dB", "dC")):
        setattr(p, n, fake(10 + i))
    for k, v in kw.items():
        if k.startswith("fwd_"):
            setattr(p.fwd, k[4:], v)
        else:
            setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    ({"fwd_disc": _lib.SSM_DISC_ZOH}, _lib.SSM_ERR_UNSUPPORTED),
    ({"fwd_dstate": 96}, _lib.SSM_ERR_UNSUPPORTED),
    ({"ddt": None}, _lib.SSM_ERR_INVALID_ARG),
    ({"fwd_z": fake(20)}, _lib.SSM_ERR_INVALID_ARG),
    ({"fwd_dt_bias": fake(20)}, _lib.SSM_ERR_INVALID_ARG),
    ({"dB": FAKE + 4}, _lib.SSM_ERR_INVALID_ARG),
])
def test_ssd_bwd_rejects_bad_arguments(lib, kw, status):
    p = ssd_bwd_params(**kw)
    assert lib.ssd_scan_bwd(ctypes.byref(p), fake(30), 1 << 40, None) == status
    assert lib.ssm_last_error()


def chunked_bwd_workspace_bytes(batch, L, H, P, N, es=2):
    """The chunked SSD backward's scratch: chunk states and adjoints ([P][N] float32 per
    64-step chunk) for one slice of (batch, head) sequences, the slice as large as fits
    in the bytes of x and dy and then evened out over the slices; a chunk sum of dt A and
    three per-chunk partial sums for every sequence; each part rounded up to 256 bytes."""
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    nch, seqs = -(-L // 64), batch * H
    nq = min(seqs, max(1, (2 * batch * L * H * P * es) // (2 * nch * P * N * 4)))
    slices = -(-seqs // nq)
    nq = -(-seqs // slices)
    return 2 * r256(nq * nch * P * N * 4) + r256(seqs * nch * 4) + r256(3 * seqs * nch * 4)


def test_ssd_bwd_workspace_size(lib):
    p = ssd_bwd_params()  # dstate 128, headdim 64: the chunked form
    need = lib.ssd_scan_bwd_workspace_size(ctypes.byref(p))
    assert need == chunked_bwd_workspace_bytes(2, 64, 4, 64, 128)
    assert lib.ssd_scan_bwd(ctypes.byref(p), fake(30), need - 1, None) == _lib.SSM_ERR_INVALID_ARG
    p = ssd_bwd_params(fwd_headdim=16)  # outside the chunked form's shapes: the tied recurrence
    need = lib.ssd_scan_bwd_workspace_size(ctypes.byref(p))
    assert need == bwd_workspace_bytes(2 * 4 * 16, 128, 64)
    p = ssd_bwd_params(fwd_batch=3, fwd_seqlen=1000, fwd_nheads=5, fwd_in_dtype=_lib.SSM_F32,
                       fwd_out_dtype=_lib.SSM_F32)
    need = lib.ssd_scan_bwd_workspace_size(ctypes.byref(p))
    assert need == chunked_bwd_workspace_bytes(3, 1000, 5, 64, 128, es=4)
    # dy in another dtype than the inputs: the tied recurrence
    p = ssd_bwd_params(fwd_out_dtype=_lib.SSM_F32)
    need = lib.ssd_scan_bwd_workspace_size(ctypes.byref(p))
    assert need == bwd_workspace_bytes(2 * 4 * 64, 128, 64, dy_bytes=4)
    # the other chunked shapes, and one slice per sequence when x and dy are small
    for N, P in ((64, 64), (128, 32), (64, 32)):
        p = ssd_bwd_params(fwd_dstate=N, fwd_headdim=P, fwd_seqlen=130)
        assert lib.ssd_scan_bwd_workspace_size(ctypes.byref(p)) == chunked_bwd_workspace_bytes(2, 130, 4, P, N)


def test_backward_workspace_at_most_the_inputs(lib):
    """At the benchmark shapes the backward's scratch is no larger than its inputs
    (x, delta, B, C, dy, z where present)."""
    # SSD 130m: batch 4, L 4096, 24 heads x 64, dstate 128, bf16, no z
    p = ssd_bwd_params(fwd_batch=4, fwd_seqlen=4096, fwd_nheads=24, fwd_headdim=64)
    L, HP, N = 4096, 24 * 64, 128
    inputs = 4 * L * HP * 2 * 2 + 4 * L * 24 * 2 + 2 * 4 * L * N * 2
    need = lib.ssd_scan_bwd_workspace_size(ctypes.byref(p))
    assert 0 < need <= inputs
    # Mamba-1 130m layer: batch 8, d_inner 1536, dstate 16, L 2048, bf16, z
    p = scan_bwd_params(fwd_batch=8, fwd_dim=1536, fwd_seqlen=2048, fwd_z=fake(20), dz=fake(21))
    inputs = 4 * 8 * 1536 * 2048 * 2 + 2 * 8 * 16 * 2048 * 2
    need = lib.ssm_scan_bwd_workspace_size(ctypes.byref(p))
    assert 0 < need <= inputs
    # Mamba-1 790m, one row of 32768 steps
    p = scan_bwd_params(fwd_batch=1, fwd_dim=3072, fwd_seqlen=32768)
    inputs = 3 * 3072 * 32768 * 2 + 2 * 16 * 32768 * 2
    need = lib.ssm_scan_bwd_workspace_size(ctypes.byref(p))
    assert 0 < need <= inputs


