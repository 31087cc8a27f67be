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
        m.mercury_attn_sharded(q, k, v, 4, 1, False, out=torch.zeros(1, 4, 256, 128),
                               lse=torch.zeros(1, 4, 256))


def _outs(shape_o=(1, 4, 256, 128), shape_l=(1, 4, 256), dtype=torch.float32):
    return torch.zeros(shape_o, dtype=dtype), torch.zeros(shape_l)


@pytest.mark.parametrize("call", ["sharded", "sharded_bf16", "split_noalloc", "decode", "run_schedule",
                                  "tune_schedule"])
@pytest.mark.parametrize("which", ["out", "lse"])
def test_undersized_outputs_rejected_before_the_library(m, monkeypatch, call, which):
    """A caller-provided out or lse smaller (or larger) than [B,Hq,Sq,d] /
    [B,Hq,Sq] would be written past its end: the binding refuses it before
    any pointer reaches the library."""
    def no_call(*a, **kw):
        raise AssertionError("the library was called")
    monkeypatch.setattr(m, "lib", type("NoLib", (), {n: staticmethod(no_call) for n in m.EXPORTED})())
    q, k, v = _qkv()
    dt = torch.bfloat16 if call == "sharded_bf16" else torch.float32
    out, lse = _outs(dtype=dt)
    if which == "out":
        out = torch.zeros((1, 4, 255, 128), dtype=dt)
    else:
        lse = torch.zeros((1, 4, 128))
    fn = {"sharded": lambda: m.mercury_attn_sharded(q, k, v, 4, 1, False, out, lse),
          "sharded_bf16": lambda: m.mercury_attn_sharded_bf16(q, k, v, 4, 1, False, out, lse),
          "split_noalloc": lambda: m.mercury_attn_split_noalloc(q, k, v, 4, 1, False, 2, out, lse),
          "decode": lambda: m.mercury_attn_decode(q, k, v, 0, False, out, lse),
          "run_schedule": lambda: m.mercury_attn_run_schedule(q, k, v, False, (4, 4, 1, 1), out, lse),
          "tune_schedule": lambda: m.mercury_tune_schedule(q, k, v, 4, 1, False, 0, 2, out, lse)}[call]
    with pytest.raises(ValueError, match="%s must have shape" % which):
        fn()


def test_partial_and_merge_output_shapes_checked(m):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="o_part must have shape"):
        m.mercury_attn_partial(q, k, v, 4, 1, False, torch.zeros(3, 1, 4, 256, 128), torch.zeros(4, 1, 4, 256))
    with pytest.raises(ValueError, match="lse_part must have shape"):
        m.mercury_attn_partial(q, k, v, 4, 1, False, torch.zeros(4, 1, 4, 256, 128), torch.zeros(4, 1, 4, 255))
    o = torch.zeros(4, 10, 128)
    lp = torch.zeros(4, 10)
    with pytest.raises(ValueError, match="out must hold"):
        m.mercury_lse_merge(o, lp, torch.zeros(9, 128), torch.zeros(10))
    with pytest.raises(ValueError, match="lse must hold"):
        m.mercury_lse_merge(o, lp, torch.zeros(10, 128), torch.zeros(9))
    with pytest.raises(ValueError, match="c must have shape"):
        m.mercury_gemm_shifted(torch.zeros(16, 8, dtype=torch.bfloat16), torch.zeros(8, 32, dtype=torch.bfloat16),
                               2, 1, torch.zeros(16, 31))


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


@pytest.mark.gpu
def test_default_stream_pointer_is_the_current_stream(m):
    """Calls without stream= run on the caller's current stream: the raw
    stream getter gives the same handle as torch's public current_stream(),
    on the default stream and inside a stream context."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert m._stream_ptr(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert m._stream_ptr(None) == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert m._stream_ptr(None) == torch.cuda.current_stream().cuda_stream
    assert m._stream_ptr(s) == s.cuda_stream
    assert m._stream_ptr(s.cuda_stream) == s.cuda_stream
