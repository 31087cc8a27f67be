"""The Python binding's argument marshalling, without a GPU: it refuses
tensors the C ABI cannot take (CPU memory, wrong dtype, non-contiguous,
mismatched shapes) before any library call, and maps status codes to
MercuryError with the library's message."""
import ctypes

import pytest
import torch


@pytest.fixture(scope="module")
def m():
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury
    return mercury


def _qkv(dtype=torch.bfloat16, device="cpu"):
    q = torch.zeros(1, 4, 256, 128, dtype=dtype, device=device)
    k = torch.zeros(1, 2, 256, 128, dtype=dtype, device=device)
    return q, k, k.clone()


def test_cpu_tensors_rejected(m):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA"):
        m.mercury_attn_sharded(q, k, v, 4, 1, False, out=torch.zeros(1), lse=torch.zeros(1))


def test_shape_mismatch_rejected(m):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="shape mismatch"):
        m.mercury_attn_sharded(q, k, v[:, :, :128], 4, 1, False)
    with pytest.raises(ValueError, match="4-D"):
        m.mercury_attn_sharded(q[0], k, v, 4, 1, False)


def test_dtype_and_layout_checks(m):
    t = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="CUDA"):
        m._dev_ptr(t, "torch.float32", "x")
    with pytest.raises(TypeError, match="torch tensor"):
        m._dev_ptr([1, 2], "torch.float32", "x")


def test_status_codes_map_to_mercury_error(m):
    # a planner call that fails validation: the message of the library comes along
    with pytest.raises(m.MercuryError) as e:
        m.mercury_plan_shift(8, 3)
    assert e.value.status == m.MERCURY_EINVAL
    assert "nested shift" in str(e.value)
    assert m.lib.mercury_last_error()


def test_status_names_cover_header_codes(m):
    import os
    import re
    from tests.conftest import ROOT
    text = open(os.path.join(ROOT, "include", "mercury_attn.h")).read()
    codes = dict((name, int(val)) for name, val in re.findall(r"#define (MERCURY_E\w+)\s+\((-?\d+)\)", text))
    assert codes, "no status codes found"
    for name, val in codes.items():
        assert getattr(m, name) == val, name
        assert val in m._STATUS_NAMES, name


def _header_struct_fields(name):
    import os
    import re
    from tests.conftest import ROOT
    text = open(os.path.join(ROOT, "include", "mercury_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (name, name), text, flags=re.S).group(1)
    return [(t, n) for t, n in re.findall(r"(double|int|long long)\s+(\w+);", body)]


def test_structs_match_header(m):
    """The ctypes mirrors of mercury_schedule and mercury_cost_profile have the
    header's fields, in order, with matching C types."""
    ctype = {"double": ctypes.c_double, "int": ctypes.c_int, "long long": ctypes.c_longlong}
    for cname, py in (("mercury_schedule", m.Schedule), ("mercury_cost_profile", m.CostProfile)):
        fields = _header_struct_fields(cname)
        assert fields, cname
        assert [(n, ctype[t]) for t, n in fields] == list(py._fields_), cname
