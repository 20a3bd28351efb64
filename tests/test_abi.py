"""The C-ABI library loads and exports every symbol include/rx.h declares; host
argument validation rejects bad calls before touching a device (CPU only)."""
import ctypes
import os
import re

import pytest

from tests._util import LIB, ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "rx.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rx_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    try:
        ensure_built()
    except RuntimeError as e:  # pragma: no cover
        pytest.skip("cannot build librx.so here: %s" % e)
    return ctypes.CDLL(LIB)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), "librx.so does not export %s" % n
    from partitioned_kv_cache_gb300 import rx
    assert sorted(rx.EXPORTS) == names


def test_status_strings(lib):
    lib.rx_status_str.restype = ctypes.c_char_p
    assert lib.rx_status_str(0) == b"RX_OK"
    assert lib.rx_status_str(-3) == b"RX_ERR_CAPACITY"
    assert lib.rx_status_str(-99) == b"RX_ERR_UNKNOWN"


def test_create_rejects_bad_configs_without_a_device(lib):
    from partitioned_kv_cache_gb300 import rx
    h = ctypes.c_void_p()
    bad = [
        rx.RxConfig(0, 8, 1, 256, 64, 8, 256, 51, 0, 0, 0),     # L = 0
        rx.RxConfig(1, 8, 3, 256, 64, 8, 256, 51, 0, 0, 0),     # Hq % Hkv
        rx.RxConfig(1, 8, 1, 96, 64, 8, 256, 51, 0, 0, 0),      # D
        rx.RxConfig(1, 8, 1, 256, 64, 0, 256, 51, 0, 0, 0),     # N = 0
        rx.RxConfig(1, 8, 1, 256, -1, 8, 256, 51, 0, 0, 0),     # P_cap < 0
        rx.RxConfig(1, 6, 1, 256, 64, 8, 256, 51, 0, 0, 0),     # G = 6 not a power of two
    ]
    for cfg in bad:
        st = rx._lib.rx_cache_create(ctypes.byref(cfg), ctypes.byref(h))
        assert st in (-1, -6), st
        assert h.value is None
    assert rx._lib.rx_cache_create(None, ctypes.byref(h)) == -1


def test_norm_and_gamma_reject_bad_arguments(lib):
    from partitioned_kv_cache_gb300 import rx
    L = rx._lib
    buf = ctypes.create_string_buffer(4096 + 16)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert L.rx_adarmsnorm(p, p, 4, 7, 1e-6, p + 1024, None) == -1       # d % 8
    assert L.rx_adarmsnorm(p, p, -1, 8, 1e-6, p + 1024, None) == -1      # rows < 0
    assert L.rx_adarmsnorm(p, p, 4, 8, 1e-6, p, None) == -1              # alias
    assert L.rx_adarmsnorm(p + 2, p, 4, 8, 1e-6, p + 1024, None) == -1   # misaligned
    assert L.rx_adarmsnorm(p, p, 0, 8, 1e-6, p + 1024, None) == 0        # empty: no-op
    assert L.rx_ada_gamma(p, p, 0, 16, 16, p, p, 64, p, p, 128, 1, p, None) == -1     # n_cond
    assert L.rx_ada_gamma(p, p, 17, 16, 16, p, p, 64, p, p, 128, 1, p, None) == -1    # n_cond
    assert L.rx_ada_gamma(p, p, 1, 15, 16, p, p, 64, p, p, 128, 1, p, None) == -1     # odd emb
    assert L.rx_ada_gamma(p, p, 1, 16, 16, p, p, 60, p, p, 128, 1, p, None) == -1     # hidden % 16
    assert L.rx_ada_gamma(p, p, 1, 16, 16, p, p, 72, p, p, 128, 1, p, None) == -1     # hidden % 16
    assert L.rx_ada_gamma(p, p, 1, 16, 16, p, p, 64, p, p, 100, 1, p, None) == -1     # d % 8
    assert L.rx_ada_gamma(p, p, 1, 16, 16, p, p, 64, p, p, 128, 0, p, None) == -1     # n_sets
    L.rx_last_error.restype = ctypes.c_char_p
    assert b"n_sets" in L.rx_last_error()


def test_cache_calls_reject_null_handle(lib):
    from partitioned_kv_cache_gb300 import rx
    L = rx._lib
    assert L.rx_cache_destroy(None) == 0
    assert L.rx_pin_prefix(None, None, None, 0, None) == -1
    assert L.rx_push_frame(None, None, None, None, None) == -1
    assert L.rx_attend_suffix(None, 0, None, None, None, 1, None, None) == -1
    assert L.rx_attend_batch(None, 0, None, None, None, 0, None, None, None) == -1
    assert L.rx_set_attn_splits(None, 0) == -1
    assert L.rx_set_attn_dparts(None, 0) == -1
    assert L.rx_debug_inject_timeout(None, 16) == -1


def test_binding_checks_tensors_before_calling_the_library(lib):
    """rx.py only marshals arguments: a wrong dtype, a strided view or a host
    tensor is refused in Python, before any C call (CPU only)."""
    import torch
    from partitioned_kv_cache_gb300 import rx
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    g = torch.ones(64, dtype=torch.float32)
    with pytest.raises(TypeError):
        rx.adarmsnorm(x.float(), g, 1e-6)                  # fp32 input
    with pytest.raises(ValueError):
        rx.adarmsnorm(torch.zeros(64, 8, dtype=torch.bfloat16).t(), g, 1e-6)   # not contiguous
    with pytest.raises(ValueError):
        rx.adarmsnorm(x, g, 1e-6)                          # host memory
    with pytest.raises(rx.RxError):
        rx.choose_partition(34, 4, 96, 152, 64, [0] * 17)  # head dimension 96


def test_binding_refuses_shapes_the_library_would_overrun(lib):
    """Sizes passed to the library come from the tensors' shapes; a tensor of
    another shape (a shorter V, a smaller output, another head count) is
    refused in Python before any C call, so the kernels never read or write
    past a caller's buffer (CPU only: host tensors, no cache handle)."""
    import torch
    from partitioned_kv_cache_gb300 import rx
    bf = dict(dtype=torch.bfloat16)
    q = torch.zeros(5, 8, 64, **bf)
    k = torch.zeros(7, 1, 64, **bf)
    out = torch.zeros(5, 8, 64, **bf)
    static = rx.attend_regions_static
    with pytest.raises(ValueError, match="v_pin"):
        static(q, k, k[:6], None, None, None, None, out)                 # shorter V
    with pytest.raises(ValueError, match="k_win"):
        static(q, k, k, torch.zeros(7, 2, 64, **bf), torch.zeros(7, 2, 64, **bf), None, None, out)
    with pytest.raises(ValueError, match="k_dyn"):
        static(q, None, None, None, None, torch.zeros(3, 1, 128, **bf), torch.zeros(3, 1, 128, **bf), out)
    with pytest.raises(ValueError, match="out"):
        static(q, k, k, None, None, None, None, out[:4])                  # smaller output
    with pytest.raises(ValueError, match="both"):
        static(q, k, None, None, None, None, None, out)
    with pytest.raises(ValueError, match="gamma"):
        rx.adarmsnorm(torch.zeros(4, 64, **bf), torch.ones(32), 1e-6)
    with pytest.raises(ValueError, match="y"):
        rx.adarmsnorm(torch.zeros(4, 64, **bf), torch.ones(64), 1e-6, out=torch.zeros(3, 64, **bf))
    with pytest.raises(ValueError, match="v_new"):
        rx.tail_append(torch.zeros(2, 4, 1, 64, **bf), torch.zeros(2, 4, 1, 64, **bf),
                       torch.zeros(2, dtype=torch.int32), torch.zeros(2, 1, 64, **bf),
                       torch.zeros(1, 1, 64, **bf))
    W1 = torch.zeros(2, 64, 32, **bf)
    with pytest.raises(ValueError, match="W2"):
        rx.ada_gamma(torch.zeros(3), torch.zeros(3, 16), W1, torch.zeros(2, 64, **bf),
                     torch.zeros(2, 128, 32, **bf), torch.zeros(2, 128, **bf), 16)
    # The cache's calls check against its configuration (no device needed).
    c = rx.Cache.__new__(rx.Cache)
    c.cfg = rx.RxConfig(2, 8, 1, 64, 16, 4, 32, 51, 8, 4, 0)
    c._h = None
    with pytest.raises(ValueError, match="k_dyn"):
        c.attend_suffix(0, torch.zeros(5, 8, 64, **bf), torch.zeros(4, 1, 64, **bf), torch.zeros(5, 1, 64, **bf))
    with pytest.raises(ValueError, match="q"):
        c.attend_suffix(0, torch.zeros(5, 4, 64, **bf), torch.zeros(5, 1, 64, **bf), torch.zeros(5, 1, 64, **bf))
    with pytest.raises(ValueError, match="out"):
        c.attend_suffix(0, q, q[:, :1].contiguous(), q[:, :1].contiguous(), out=out[:, :4].contiguous())
    with pytest.raises(ValueError, match="k"):
        c.push_frame(torch.zeros(2, 31, 1, 64, **bf), torch.zeros(2, 31, 1, 64, **bf))
    with pytest.raises(ValueError, match="v"):
        c.pin_prefix(torch.zeros(2, 16, 1, 64, **bf), torch.zeros(2, 15, 1, 64, **bf))
    with pytest.raises(ValueError, match="k_tail"):
        c.attend_batch(0, None, (torch.zeros(4, 1, 8, 64, **bf), torch.zeros(4, 7, 1, 64, **bf),
                                 torch.zeros(4, 7, 1, 64, **bf), torch.zeros(4, dtype=torch.int32)))
