"""The C ABI library: it loads, exports every declared entry point, and rejects bad
arguments on the host before touching CUDA (CPU only, no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_39_gb300 import _build
    import gated_delta_rule_39_gb300 as kda
    _build.build()
    return kda.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("kda_fwd", "kda_fwd_host", "kda_fwd_get_error", "kda_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from gated_delta_rule_39_gb300 import _build
    nm = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s(\w+)$", nm, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings(lib):
    import gated_delta_rule_39_gb300 as kda
    assert kda.kda_status_string(0) == "KDA_OK"
    for code in range(-1, -14, -1):
        assert kda.kda_status_string(code).startswith("KDA_ERR_")
    assert "unknown" in kda.kda_status_string(12345)


def _call(lib, **over):
    """Call kda_fwd with fake (never dereferenced) pointers; host validation only."""
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, k=fake, v=fake, g=fake, beta=ctypes.c_void_p(0x90000), scale=0.1,
             out=ctypes.c_void_p(0x80000000), A_log=fake, dt_bias=fake, lower_bound=-5.0,
             s0=None, s0_dtype=0, s1=None, s1_dtype=0, cu=None, num_seqs=0, B=1, T=16, H=1,
             K=128, V=128)
    a.update(over)
    return lib.kda_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["out"],
                       a["A_log"], a["dt_bias"], a["lower_bound"], a["s0"], a["s0_dtype"],
                       a["s1"], a["s1_dtype"], a["cu"], a["num_seqs"], a["B"], a["T"], a["H"],
                       a["K"], a["V"], None)


def test_rejects_unsupported_dims(lib):
    assert _call(lib, K=64) == -3
    assert _call(lib, V=256) == -3


def test_rejects_bad_shapes(lib):
    assert _call(lib, B=0) == -2
    assert _call(lib, T=-1) == -2
    assert _call(lib, H=0) == -2
    assert _call(lib, cu=ctypes.c_void_p(0x20000), num_seqs=0) == -2
    assert _call(lib, cu=ctypes.c_void_p(0x20000), num_seqs=2, B=2) == -2
    assert _call(lib, T=1 << 20, H=64) == -2      # 2^33 elements


def test_rejects_null_pointers(lib):
    assert _call(lib, q=None) == -1
    assert _call(lib, out=None) == -1
    assert _call(lib, A_log=None) == -1


def test_rejects_bad_dtypes_and_args(lib):
    fake = ctypes.c_void_p(0x7000000)
    assert _call(lib, s0=fake, s0_dtype=7) == -5
    assert _call(lib, s1=fake, s1_dtype=-1) == -5
    assert _call(lib, lower_bound=-6.0) == -12
    assert _call(lib, lower_bound=-5.45) == -12
    assert _call(lib, lower_bound=0.5) == -12
    assert _call(lib, scale=float("inf")) == -12


def test_rejects_misaligned_pointers(lib):
    assert _call(lib, q=ctypes.c_void_p(0x10008)) == -4
    assert _call(lib, out=ctypes.c_void_p(0x80000002)) == -4


def test_rejects_aliasing(lib):
    assert _call(lib, out=ctypes.c_void_p(0x10000)) == -13
    # states of different dtypes in one buffer
    s = ctypes.c_void_p(0x7000000)
    assert _call(lib, s0=s, s0_dtype=0, s1=s, s1_dtype=1) == -13


def test_workspace_size(lib):
    import gated_delta_rule_39_gb300 as kda
    assert kda.kda_fwd_workspace_bytes(1, 0, 4) == 0
    assert kda.kda_fwd_workspace_bytes(1, 8192, 96) == 0          # fixed length: none
    assert kda.kda_fwd_workspace_bytes(1, 8192, 96, 12, True) >= 4 * 13


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gated_delta_rule_39_gb300 as kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        kda.load_library()


def test_last_cuda_error_reports_missing_device():
    """With every GPU hidden, a well-formed call fails in the CUDA runtime before any
    launch: KDA_ERR_CUDA, and kda_last_cuda_error names the runtime's error."""
    code = (
        "import ctypes, test_abi as t\n"
        "import gated_delta_rule_39_gb300 as kda\n"
        "lib = kda.load_library()\n"
        "assert kda.kda_last_cuda_error() == 0\n"
        "rc = t._call(lib)\n"
        "print(rc, kda.kda_last_cuda_error())\n"
    )
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="",
               PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests")]))
    from gated_delta_rule_39_gb300 import _build
    _build.build()
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    rc, cuda_err = map(int, r.stdout.split())
    assert rc == -11            # KDA_ERR_CUDA
    assert cuda_err != 0        # cudaErrorNoDevice (or another "no device" code)
