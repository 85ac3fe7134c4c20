"""The C-ABI library on the host: it loads without a GPU, exports every
symbol include/attn.h declares, and rejects bad arguments before launching
anything."""
import ctypes
import re
import os

import pytest

from exact_tiled_attention_online_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/attn.h but not exported"


def test_version_and_strings(lib):
    assert lib.attn_version() >= 100
    for code in range(9):
        assert attn.status_string(code)


def _fwd(lib, **over):
    args = dict(q=1, k=1, v=1, o=1, lse=1, o_f32=None, cu_q=1, cu_k=1, batch=1, max_q=4, max_k=4,
                total_q=4, total_k=4, hq=2, hkv=1, d=64, scale=0.125, mask=1, window=0, slopes=None, dtype=0,
                ws=None, ws_bytes=0, stream=None)
    args.update(over)
    return lib.attn_fwd(*args.values())


@pytest.mark.parametrize("over,code", [
    ({"hq": 3, "hkv": 2}, 1),            # Hq not a multiple of Hkv
    ({"hkv": 0}, 1),
    ({"d": 96}, 2),                      # head_dim not built
    ({"batch": -1}, 1),
    ({"total_q": -5}, 1),
    ({"max_q": 8}, 1),                   # max_seqlen above total
    ({"mask": 7}, 1),
    ({"window": -1}, 1),                 # negative window
    ({"mask": 0, "window": 4}, 1),       # a window needs a causal rule
    ({"dtype": 9}, 1),
    ({"scale": float("nan")}, 1),
    ({"scale": float("inf")}, 1),
    ({"q": None}, 1),
    ({"cu_q": None}, 1),
])
def test_fwd_rejects_bad_arguments(lib, over, code):
    assert _fwd(lib, **over) == code


def test_workspace_size_rejects_bad_arguments(lib):
    assert lib.attn_fwd_workspace_size(1, 4, 4, 4, 3, 2, 64, 0, 0) == ctypes.c_size_t(-1).value
    assert lib.attn_fwd_workspace_size(1, 4, 4, 4, 2, 1, 64, -3, 0) == ctypes.c_size_t(-1).value
    assert lib.attn_bwd_workspace_size(1, 4, 4, 4, 4, 2, 1, 80, 0) == ctypes.c_size_t(-1).value


def test_bwd_workspace_covers_rows_and_fp16_copies(lib):
    n = lib.attn_bwd_workspace_size(2, 100, 100, 200, 200, 4, 2, 128, 0)
    rows = 2 * 4 * 200 * 4                         # D and lse2
    copies = 2 * 200 * 4 * 128 * 2 + 2 * 200 * 2 * 128 * 2   # q, dout, k, v in fp16
    assert n >= rows + copies
    assert lib.attn_bwd_workspace_size(2, 100, 100, 200, 200, 4, 2, 128, 1) >= rows
    # head_dim 128 bf16 also holds the fused backward's fp32 dQ accumulator
    assert n >= rows + copies + 200 * 4 * 128 * 4
    n64 = lib.attn_bwd_workspace_size(2, 100, 100, 200, 200, 4, 2, 64, 0)
    copies64 = copies // 2
    assert rows + copies64 <= n64 < rows + copies64 + 200 * 4 * 64 * 4  # head_dim 64: no accumulator


def test_deterministic_switch_round_trips(lib):
    """The backward-form switch is process-wide host state: set, read back,
    restored (no device needed)."""
    prev = attn.get_deterministic()
    try:
        attn.set_deterministic(True)
        assert attn.get_deterministic() is True
        assert lib.attn_get_deterministic() == 1
        attn.set_deterministic(False)
        assert attn.get_deterministic() is False
        lib.attn_set_deterministic(7)  # any nonzero value selects the two-kernel form
        assert lib.attn_get_deterministic() == 1
    finally:
        attn.set_deterministic(prev)


def test_bwd_rejects_missing_workspace(lib):
    st = lib.attn_bwd(1, 1, 1, 1, 1, None, 1, 1, 1, 1, 1, 1, 1, 4, 4, 4, 4, 2, 1, 64, 0.1, 1, 0,
                      None, 0, None, 0, None)
    assert st == 3


def test_bwd_rejects_window_without_causal_rule(lib):
    st = lib.attn_bwd(1, 1, 1, 1, 1, None, 1, 1, 1, 1, 1, 1, 1, 4, 4, 4, 4, 2, 1, 64, 0.1, 0, 5,
                      None, 0, None, 0, None)
    assert st == 1


def test_probe_rejects_bad_tile_rows(lib):
    assert lib.attn_mask_probe(1, 1, 1, 4, 4, 4, 4, 1, 0, 48, 1, None) == 1
    assert lib.attn_mask_probe(1, 1, 1, 4, 4, 4, 4, 1, -2, 128, 1, None) == 1


def test_strided_entry_rejects_bad_strides(lib):
    """A token stride of 3 elements (6 bytes) breaks the 16-byte rule."""
    s = attn.AttnStrides()
    s.k[0], s.k[1] = 64, 64   # valid: contiguous [T, 1, 64]
    s.v[0], s.v[1] = 64, 64
    s.o[0], s.o[1] = 128, 64
    s.q[0], s.q[1] = 3, 64    # invalid: 6 bytes
    lib.attn_fwd_ex.argtypes = ([ctypes.POINTER(attn.AttnStrides), ctypes.POINTER(attn.AttnBiasTensor)]
                                + lib.attn_fwd.argtypes)
    args = dict(q=1, k=1, v=1, o=1, lse=1, o_f32=None, cu_q=1, cu_k=1, batch=1, max_q=4,
                max_k=4, total_q=4, total_k=4, hq=2, hkv=1, d=64, scale=0.125, mask=1, window=0,
                slopes=None, dtype=0, ws=None, ws_bytes=0, stream=None)
    assert lib.attn_fwd_ex(ctypes.byref(s), None, *args.values()) == 1
    s.q[0] = 0  # only positive strides
    assert lib.attn_fwd_ex(ctypes.byref(s), None, *args.values()) == 1


def test_bias_tensor_rejections(lib):
    """A bias tensor without data, with a negative stride or misaligned data
    is refused before any launch."""
    ex = [ctypes.POINTER(attn.AttnStrides), ctypes.POINTER(attn.AttnBiasTensor)]
    lib.attn_fwd_ex.argtypes = ex + lib.attn_fwd.argtypes
    lib.attn_bwd_ex.argtypes = ex + lib.attn_bwd.argtypes
    fargs = [1, 1, 1, 1, 1, None, 1, 1, 1, 4, 4, 4, 4, 2, 1, 64, 0.125, 1, 0, None, 0, None, 0, None]
    bargs = [1] * 10 + [1, 1, 1, 4, 4, 4, 4, 2, 1, 64, 0.125, 1, 0, None, 0, None, 0, None]
    for data, strides in ((None, (0, 0, 4)), (256, (0, -1, 4)), (256, (-4, 0, 4)),
                          (256, (0, 0, -4)), (258, (0, 0, 4))):
        b = attn.AttnBiasTensor(data, *strides)
        assert lib.attn_fwd_ex(None, ctypes.byref(b), *fargs) == 1
        assert lib.attn_bwd_ex(None, ctypes.byref(b), *bargs) == 1


@pytest.mark.parametrize("shape,err", [((2, 4, 8, 8), "CUDA"), ((8, 8), "CUDA")])
def test_binding_refuses_host_or_misshapen_bias(shape, err):
    """The binding refuses a bias that is not a CUDA fp32 tensor before any
    call into the library."""
    import torch
    with pytest.raises(ValueError, match=err):
        attn._btab(torch.zeros(shape), 2, 4, 8, 8)


def test_binding_bias_strides_broadcast():
    """Broadcast dimensions (size 1) get stride 0; the key stride must be 1.
    Checked on the stride arithmetic alone, with a stand-in for the tensor."""
    class FakeTensor:  # quacks like a CUDA fp32 tensor for _btab's checks
        import torch
        is_cuda, dtype = True, torch.float32

        def __init__(self, shape, strides):
            self.shape, self._st = shape, strides

        def dim(self):
            return len(self.shape)

        def stride(self, i):
            return self._st[i]

        def data_ptr(self):
            return 4096

    b = attn._btab(FakeTensor((1, 4, 8, 9), (288, 72, 9, 1)), 2, 4, 8, 9)
    assert (b.seq_stride, b.head_stride, b.row_stride) == (0, 72, 9)
    b = attn._btab(FakeTensor((2, 1, 8, 9), (72, 0, 9, 1)), 2, 4, 8, 9)
    assert (b.seq_stride, b.head_stride, b.row_stride) == (72, 0, 9)
    with pytest.raises(ValueError):
        attn._btab(FakeTensor((2, 4, 8, 9), (288, 72, 1, 8)), 2, 4, 8, 9)  # keys not contiguous
    with pytest.raises(ValueError):
        attn._btab(FakeTensor((2, 4, 7, 9), (252, 63, 9, 1)), 2, 4, 8, 9)  # too few rows
    with pytest.raises(ValueError):
        attn._btab(FakeTensor((3, 4, 8, 9), (288, 72, 9, 1)), 2, 4, 8, 9)  # wrong batch
