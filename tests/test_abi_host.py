"""Host-only checks of the boundary: the library builds, loads and exports every
entry point that include/zero_gb300.h declares (no compute call, no GPU)."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"ZERO_API\s+[\w\s\*]*?\b(zero_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from zero_partitioned_mixed_gb300.build import build_library
    build_library()
    import zero_partitioned_mixed_gb300 as Z
    return Z


def test_header_declares_the_boundary():
    names = _declared()
    assert {"zero_init_partition", "zero_step", "zero_gather_bucket", "zero_reduce_scatter_bucket",
            "zero_bytes_moved", "zero_get_status", "zero_partition_info", "zero_set_scaler",
            "zero_last_error", "zero_destroy"} <= names


def test_library_exports_every_declared_symbol(lib):
    import ctypes
    so = ctypes.CDLL(lib.library_path())
    for name in _declared():
        assert hasattr(so, name), name
    assert set(lib.exported_symbols()) == set(lib._binding.EXPORTS)


def test_library_hides_internal_symbols(lib):
    import ctypes
    so = ctypes.CDLL(lib.library_path())
    # only the C entry points are visible; launch helpers stay internal
    assert not hasattr(so, "_ZN2zg6launchENS_4KindEibRKNS_4ArgsEP11CUstream_stPi")


def test_init_errors_without_gpu_are_codes_not_crashes(lib):
    # argument errors are found before any CUDA call
    with pytest.raises(lib.ZeroError) as e:
        lib.zero_init_partition(10, 0, 1, lib.ZERO_BF16)
    assert e.value.code == 1 and "n_ranks" in str(e.value)
    with pytest.raises(lib.ZeroError) as e:
        lib.zero_init_partition(10, 2, 7, lib.ZERO_BF16)
    assert e.value.code == 1
    with pytest.raises(lib.ZeroError) as e:
        lib.zero_init_partition(10, 2, 0, lib.ZERO_BF16, 8, lib.ZERO_F_DOUBLE_BUFFER)
    assert e.value.code == 1
    with pytest.raises(lib.ZeroError) as e:
        lib.zero_init_partition(10, 65, 1, lib.ZERO_FP16)
    assert e.value.code == 1


def test_null_handle_calls_return_einval(lib):
    so = lib.load_library()
    assert so.zero_step(None, None, None, None, None, None, None, None) == 1
    assert so.zero_get_status(None, None, None) == 1
    assert so.zero_bytes_moved(None, None) == 1
    so.zero_destroy(None)
    assert b"handle" in so.zero_last_error(None)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from zero_partitioned_mixed_gb300 import _binding as B
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(B.ZeroError) as e:
        B.load_library()
    assert "build" in str(e.value)


def test_pointer_array_holds_the_rows_and_passes_through():
    # pointer_array(rows) is what every list-taking call builds internally;
    # a prebuilt array must reach the C call unchanged
    import ctypes
    import torch
    from zero_partitioned_mixed_gb300 import _binding as B
    rows = [torch.empty(16) for _ in range(5)]
    arr = B.pointer_array(rows)
    assert isinstance(arr, ctypes.Array) and len(arr) == 5
    assert [arr[i] for i in range(5)] == [t.data_ptr() for t in rows]
    assert B._ptr_array(arr) is arr
    assert B._ptr_array(None) is None


def test_noalloc_scratch_size_matches_the_header():
    # the header states the size of zero_step_noalloc's static array; the
    # library reports the size it was built with (a host query, no GPU)
    import re
    import zero_partitioned_mixed_gb300 as Z
    hdr = open(os.path.join(ROOT, "include", "zero_gb300.h")).read()
    psi_pad = int(re.search(r"#define ZERO_NOALLOC_MAX_PSI_PAD \(1ull << (\d+)\)", hdr).group(1))
    extra = [int(x.replace(",", "")) for x in re.findall(r"ZERO_NOALLOC_MAX_PSI_PAD floats plus ([\d,]+) bytes", hdr)]
    extra += [int(x.replace(",", "")) for x in re.findall(r"4 \* ZERO_NOALLOC_MAX_PSI_PAD \+ ([\d,]+)\.", hdr)]
    assert len(extra) == 2 and extra[0] == extra[1], extra
    assert Z.zero_noalloc_scratch_bytes() == 4 * (1 << psi_pad) + extra[0]
