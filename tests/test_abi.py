"""The C-ABI library loads and exports every symbol include/*.h declares (no GPU needed).

Only host-side logic is called here: the chooser, status strings, argument
checks that fail before any CUDA call.
"""

import ctypes
import glob
import os
import re

import pytest

from oracle import dpsgd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dp_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from differentially_private_gb300 import build as bld
    bld.build()
    import differentially_private_gb300 as dp
    return dp.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("dp_register_layer", "dp_norm_accumulate", "dp_clip_factors",
                     "dp_clipped_noisy_grad", "dp_create", "dp_step_status", "dp_philox_normals"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "differentially_private_gb300", "libdpclip.so"))
    for name in _declared_functions():
        assert hasattr(raw, name), name


def test_binding_names_match_header():
    import differentially_private_gb300 as dp
    assert sorted(dp.EXPORTS) == _declared_functions()
    for name in dp.EXPORTS:
        assert callable(getattr(dp, name))


def test_chooser_host_matches_oracle(lib):
    import differentially_private_gb300 as dp
    cases = [(1, 1, 1), (3, 2, 4), (3, 3, 3), (3, 5, 2), (16, 64, 32), (128, 768, 8), (128, 8, 768),
             (512, 4096, 4096), (1, 1024, 4096), (2048, 4096, 16), (2048, 16, 14336), (2048, 14336, 4096),
             (2 ** 31, 2 ** 31, 2 ** 31), (2 ** 31, 2 ** 31, 2 ** 31 + 1), (2 ** 40, 2 ** 40, 2 ** 40 + 1),
             (3037000500, 3037000500, 3037000500)]
    for n in (7, 4096, 65535):
        cases += [(n, n * n + 1, 1), (n, n * n - 1, 1), (n, n * n, 1), (n, 1, n * n + 1)]
    for T, di, do in cases:
        assert dp.dp_choose_path(T, di, do) == dpsgd.choose_path(T, di, do), (T, di, do)
    assert dp.dp_choose_path(0, 1, 1) == -1
    assert dp.dp_choose_path(1, 0, 1) == -1


def test_status_strings_and_version(lib):
    import differentially_private_gb300 as dp
    assert dp.dp_version() >= 100
    for s in range(8):
        assert dp.dp_status_string(s)
    assert dp.dp_status_string(4) == "non-finite per-example norm"


def test_null_context_is_rejected(lib):
    assert lib.dp_begin_step(None, 4) == 1
    assert lib.dp_clip_factors(None, ctypes.c_float(1.0), None, None) == 1
    assert lib.dp_num_coords(None) == 0
    assert lib.dp_destroy(None) == 0
    assert lib.dp_last_error(None) == b""


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import differentially_private_gb300 as dp
    with pytest.raises(dp.DPError) as ei:
        dp.dp_create(0, None)
    assert ei.value.status in (dp.DP_ERR_CUDA, dp.DP_ERR_UNSUPPORTED)
