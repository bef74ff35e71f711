"""The C-ABI library builds for sm_103a, loads, and exports every declared entry
point; host-side argument checks return their documented codes without
touching a GPU (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

import blocked_floyd_warshall_gb300 as bsm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(bs_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    bsm.build()
    return bsm.library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("bs_smooth_upper", "bs_smooth_bounds", "bs_smooth_bounds_batched",
                     "bs_check_feasible", "bs_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", bsm.LIBRARY_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name), name


def test_python_binding_has_the_c_names():
    for name in declared_functions():
        assert hasattr(bsm, name), name


def header_constants():
    """BS_NAME = value pairs of the header's enums (values: integers and
    shifts of integers)."""
    out = {}
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"\b(BS_[A-Z0-9_]+)\s*=\s*(\d+(?:\s*<<\s*\d+)?)", text):
            a, _, b = m.group(2).partition("<<")
            out[m.group(1)] = int(a) << int(b) if b else int(a)
    return out


def test_binding_constants_match_the_header():
    consts = header_constants()
    for name in ("BS_OK", "BS_ERR_ARG", "BS_INT32_Q10", "BS_PERK", "BS_TILE_64", "BS_TILE_128",
                 "BS_SYMMETRIC", "BS_PERK_PAIRED", "BS_ONE_LAUNCH", "BS_PAIRED_ROUNDS"):
        assert name in consts, name
    for name, value in consts.items():
        if hasattr(bsm, name):
            assert getattr(bsm, name) == value, name
    bits = [v for k, v in consts.items()
            if k in ("BS_PERK", "BS_RULE_LITERAL", "BS_VALIDATE", "BS_TILE_64", "BS_TILE_128",
                     "BS_NO_LOOKAHEAD", "BS_SYMMETRIC", "BS_PERK_PAIRED", "BS_ONE_LAUNCH",
                     "BS_PAIRED_ROUNDS")]
    assert len(set(bits)) == len(bits) and all(b & (b - 1) == 0 for b in bits)   # distinct bits


def test_strerror_and_counters(lib):
    for st in range(7):
        assert isinstance(bsm.bs_strerror(st), str) and bsm.bs_strerror(st)
    assert "unknown" in bsm.bs_strerror(99)
    assert bsm.bs_launch_count() >= 0
    bsm.bs_profile_begin()
    p = bsm.bs_profile_end()
    assert all(p[k]["launches"] == 0 for k in bsm.PHASES)


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails its checks first
FAKE2 = ctypes.c_void_p(2 << 20)


@pytest.fixture(scope="module")
def no_gpu():
    """The fake-pointer calls below must stop at the host-side checks.  They run
    only where no GPU is visible, so a check that ever let one through could not
    reach a kernel."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("fake-pointer argument tests run on GPU-less hosts only")
    except ImportError:
        pass


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE2, -1, 4, None, 0), bsm.BS_ERR_ARG),                      # n < 0
    ((FAKE, FAKE2, 8, 7, None, 0), bsm.BS_ERR_ARG),                       # ld < n
    ((FAKE, FAKE2, 8, 8, None, 1 << 15), bsm.BS_ERR_ARG),                 # unknown mode bit
    ((FAKE, FAKE2, 8, 8, None, 2), bsm.BS_ERR_ARG),                       # unknown dtype
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_RULE_LITERAL), bsm.BS_ERR_ARG),     # literal needs per-round
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_TILE_64 | bsm.BS_TILE_128), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_PERK | bsm.BS_SYMMETRIC), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, 1 << 9), bsm.BS_ERR_ARG),                  # retired bit
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_PERK_PAIRED), bsm.BS_ERR_ARG),      # paired needs per-round
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_ONE_LAUNCH | bsm.BS_PERK), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_ONE_LAUNCH | bsm.BS_TILE_128), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_ONE_LAUNCH | bsm.BS_NO_LOOKAHEAD), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_PAIRED_ROUNDS | bsm.BS_PERK), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_PAIRED_ROUNDS | bsm.BS_ONE_LAUNCH), bsm.BS_ERR_ARG),
    ((FAKE, FAKE2, 8, 8, None, bsm.BS_PAIRED_ROUNDS | bsm.BS_NO_LOOKAHEAD), bsm.BS_ERR_ARG),
    ((None, FAKE2, 8, 8, None, 0), bsm.BS_ERR_ARG),                       # null U
    ((FAKE, None, 8, 8, None, 0), bsm.BS_ERR_ARG),                        # null L
    ((FAKE, FAKE, 8, 8, None, 0), bsm.BS_ERR_ARG),                        # U aliases L
    ((ctypes.c_void_p((1 << 20) + 2), FAKE2, 8, 8, None, 0), bsm.BS_ERR_ALIGN),
    ((FAKE, FAKE2, 0, 0, None, 0), bsm.BS_OK),                            # empty: no-op
    ((None, None, 0, 0, None, 0), bsm.BS_OK),
])
def test_bounds_argument_checks(lib, no_gpu, args, code):
    assert lib.bs_smooth_bounds(*args) == code


def test_other_entry_points_argument_checks(lib, no_gpu):
    assert lib.bs_smooth_upper(FAKE, -3, 4, None, 0) == bsm.BS_ERR_ARG
    assert lib.bs_smooth_upper(FAKE, 0, 0, None, 0) == bsm.BS_OK
    assert lib.bs_smooth_upper(None, 5, 5, None, 0) == bsm.BS_ERR_ARG
    # batched: stride shorter than one molecule, negative batch, empty batch
    assert lib.bs_smooth_bounds_batched(FAKE, FAKE2, 8, 8, 63, 2, None, 0) == bsm.BS_ERR_ARG
    assert lib.bs_smooth_bounds_batched(FAKE, FAKE2, 8, 8, 64, -1, None, 0) == bsm.BS_ERR_ARG
    assert lib.bs_smooth_bounds_batched(FAKE, FAKE2, 8, 8, 64, 0, None, 0) == bsm.BS_OK
    cnt = ctypes.c_longlong(-1)
    assert lib.bs_check_feasible(FAKE, FAKE2, 8, 8, None, 0, None, None) == bsm.BS_ERR_ARG
    assert lib.bs_check_feasible(FAKE, FAKE2, 8, 7, None, 0, ctypes.byref(cnt), None) == bsm.BS_ERR_ARG
    assert lib.bs_check_feasible(FAKE, FAKE2, 0, 0, None, 0, ctypes.byref(cnt), None) == bsm.BS_OK
    assert cnt.value == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises; nothing falls back to the CPU."""
    import importlib
    monkeypatch.setattr(bsm, "_lib", None)
    monkeypatch.setattr(bsm, "LIBRARY_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        bsm.library()
    monkeypatch.undo()
    importlib.reload(bsm)
