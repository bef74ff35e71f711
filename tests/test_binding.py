"""The Python binding's marshalling on the CPU (no GPU, no library call): the
geometry, dtype bits, batch stride and errors it derives from tensors, checked
against a stub in place of libbsmooth.so that records each call."""
import ctypes

import pytest
import torch

import blocked_floyd_warshall_gb300 as bsm


class DeviceView:
    """A CPU tensor presented as a CUDA one (shape, strides, dtype, pointer)."""

    def __init__(self, t):
        self.t = t
        self.shape = t.shape
        self.dtype = t.dtype
        self.is_cuda = True

    def stride(self, d=None):
        return self.t.stride() if d is None else self.t.stride(d)

    def dim(self):
        return self.t.dim()

    def data_ptr(self):
        return self.t.data_ptr()


class StubLib:
    def __init__(self, status=0):
        self.calls = []
        self.status = status

    def __getattr__(self, name):
        if not name.startswith("bs_"):
            raise AttributeError(name)

        def call(*args):
            self.calls.append((name, args))
            if name == "bs_strerror":
                return b"stub status"
            return self.status
        return call


@pytest.fixture
def stub(monkeypatch):
    lib = StubLib()
    monkeypatch.setattr(bsm, "library", lambda: lib)
    return lib


def value(x):
    return x.value if isinstance(x, (ctypes.c_void_p, ctypes.c_longlong)) else x


def test_square_matrix_geometry_and_dtype(stub):
    U = DeviceView(torch.zeros(70, 70))
    L = DeviceView(torch.zeros(70, 70))
    bsm.bs_smooth_bounds(U, L, stream=0, flags=bsm.BS_PAIRED_ROUNDS)
    name, args = stub.calls[-1]
    assert name == "bs_smooth_bounds"
    assert value(args[0]) == U.data_ptr() and value(args[1]) == L.data_ptr()
    assert args[2:4] == (70, 70)
    assert args[5] == bsm.BS_FP32 | bsm.BS_PAIRED_ROUNDS
    Ui = DeviceView(torch.zeros(70, 70, dtype=torch.int32))
    bsm.bs_smooth_upper(Ui, stream=0)
    name, args = stub.calls[-1]
    assert name == "bs_smooth_upper" and args[1:3] == (70, 70) and args[4] == bsm.BS_INT32_Q10


def test_padded_rows_give_the_leading_dimension(stub):
    base = torch.zeros(300, 305)
    U = DeviceView(base[:, :300])              # n = 300 rows of a 305-wide buffer
    L = DeviceView(torch.zeros(300, 305)[:, :300])
    bsm.bs_smooth_bounds(U, L, stream=0)
    assert stub.calls[-1][1][2:4] == (300, 305)


def test_batched_geometry(stub):
    U = DeviceView(torch.zeros(5, 64, 68)[:, :, :64])
    L = DeviceView(torch.zeros(5, 64, 68)[:, :, :64])
    bsm.bs_smooth_bounds_batched(U, L, stream=0, flags=bsm.BS_SYMMETRIC)
    name, args = stub.calls[-1]
    assert name == "bs_smooth_bounds_batched"
    assert args[2:6] == (64, 68, 64 * 68, 5)
    assert args[7] == bsm.BS_SYMMETRIC
    counts = bsm.bs_check_feasible_noalloc(U, L, stream=0)
    assert counts == [0] * 5
    assert stub.calls[-1][0] == "bs_check_feasible_noalloc" and stub.calls[-1][1][4:6] == (64 * 68, 5)


def test_raw_pointers_need_the_geometry(stub):
    with pytest.raises(ValueError):
        bsm.bs_smooth_bounds(1 << 20, 2 << 20, stream=0)
    bsm.bs_smooth_bounds(1 << 20, 2 << 20, n=10, ld=12, stream=0)
    name, args = stub.calls[-1]
    assert value(args[0]) == 1 << 20 and args[2:4] == (10, 12)
    with pytest.raises(ValueError):
        bsm.bs_smooth_bounds_batched(1 << 20, 2 << 20, n=10, ld=12, stream=0)


def test_rejected_tensors():
    with pytest.raises(ValueError):
        bsm._geometry(DeviceView(torch.zeros(8, 8).t()), None, None)   # columns not contiguous
    with pytest.raises(ValueError):
        bsm._ptr(torch.zeros(8, 8))                                     # host memory
    with pytest.raises(ValueError):
        bsm._dtype_bits(DeviceView(torch.zeros(8, 8, dtype=torch.float64)), None)


def test_status_raises(monkeypatch):
    lib = StubLib(status=bsm.BS_ERR_ARG)
    monkeypatch.setattr(bsm, "library", lambda: lib)
    with pytest.raises(bsm.BSError) as e:
        bsm.bs_smooth_bounds(DeviceView(torch.zeros(4, 4)), DeviceView(torch.zeros(4, 4)), stream=0)
    assert e.value.status == bsm.BS_ERR_ARG
