"""The C ABI library on a host without a GPU: it builds, loads, exports every
function include/ccv.h declares, and rejects bad arguments with the documented
status codes before touching the device.  Fake (never dereferenced) pointer
values are used; a call that passes validation would try to launch, so every
call here is built to fail validation or to be empty work.
"""
from __future__ import annotations

import ctypes
import os
import sys
import re
import subprocess

import pytest
import torch

from causal_depthwise_conv1d_fwd_gb300 import _lib, build

OK, NULLP, WIDTH, SIZE, STATE, ALIAS, STRIDE, RANGE, CAP, ARG = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9
A, B, C = 0x10000, 0x2000000, 0x8000000  # fake 16-byte-aligned device addresses, far apart
D, E = 0x20000000, 0x40000000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_every_declared_function_is_exported(lib):
    names = _lib.declared_functions()
    assert set(names) == {"ccv_status_string", "ccv_version", "ccv_fwd", "ccv_update",
                          "ccv_update_spec", "paged_sconv_seq_metadata", "paged_sconv_fwd",
                          "paged_sconv_fwd_with_metadata", "paged_sconv_fwd_streams"}
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        assert getattr(lib, n) is not None
    assert set(names) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code in (OK, NULLP, WIDTH, SIZE, STATE, ALIAS, STRIDE, RANGE, CAP, ARG):
        s = _lib.status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in _lib.status_string(-1000)
    assert lib.ccv_version() == 10300


def fwd(lib, **over):
    args = dict(x=A, xsd=1, xst=64, out=B, osd=1, ost=64, w=C, wsd=4, wsw=1, bias=None,
                st=C + 4096, ssl=192, ssd=1, sst=64, nl=4, sl=3, qsl=C + 8192, batch=2,
                ci=None, hi=None, dim=64, total=10, width=4, pad=-1, silu=1, err=None,
                stream=None)
    args.update(over)
    return lib.ccv_fwd(*args.values())


def test_fwd_validation(lib):
    assert fwd(lib, width=1) == WIDTH
    assert fwd(lib, width=6) == WIDTH
    assert fwd(lib, dim=-1) == SIZE
    assert fwd(lib, batch=-2) == SIZE
    assert fwd(lib, xst=-64) == STRIDE
    assert fwd(lib, sst=-1) == STRIDE
    assert fwd(lib, sl=2) == STATE
    assert fwd(lib, st=None, hi=C + 12288) == ARG
    assert fwd(lib, x=None) == NULLP
    assert fwd(lib, qsl=None) == NULLP
    assert fwd(lib, out=A + 64) == ALIAS  # overlaps x
    # empty work succeeds without launching anything
    assert fwd(lib, total=0) == OK
    assert fwd(lib, batch=0) == OK
    assert fwd(lib, dim=0) == OK
    assert fwd(lib, total=0, x=None, out=None) == OK


def test_fwd_valid_call_reports_cuda_error_without_gpu(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-device error path")
    status = fwd(lib)
    assert status > 0  # a cudaError_t from the failed launch
    assert _lib.status_string(status)


def upd(lib, **over):
    args = dict(x=A, xsb=64, xsd=1, xst=1, out=A, osb=64, osd=1, ost=1, w=C, wsd=4, wsw=1,
                bias=None, st=B, ssl=192, ssd=1, sst=64, nl=8, sl=3, idx=None, batch=4, dim=64,
                seqlen=1, width=4, pad=-1, silu=1, err=None, stream=None)
    args.update(over)
    return lib.ccv_update(*args.values())


def test_update_validation(lib):
    assert upd(lib, width=7) == WIDTH
    assert upd(lib, seqlen=-1) == SIZE
    assert upd(lib, ssd=-1) == STRIDE
    assert upd(lib, seqlen=2, sl=3) == STATE  # needs W-2+seqlen = 4 columns
    assert upd(lib, sl=2) == STATE
    assert upd(lib, st=None) == NULLP
    assert upd(lib, out=A + 2) == ALIAS  # overlapping but not identical to x
    assert upd(lib, batch=0) == OK
    assert upd(lib, seqlen=0) == OK


def upd_spec(lib, **over):
    args = dict(x=A, xsb=256, xsd=1, xst=64, out=A, osb=256, osd=1, ost=64, w=C, wsd=4, wsw=1,
                bias=None, st=B, ssl=448, ssd=1, sst=64, nl=32, sl=7, idx=None, nacc=None,
                inter=None, isb=0, ist=0, isd=0, isw=0, isteps=0, oidx=None, oisb=0, oist=0,
                osteps=0, batch=4, dim=64, seqlen=4, width=4, pad=-1, silu=1, err=None,
                stream=None)
    args.update(over)
    return lib.ccv_update_spec(*args.values())


def test_update_spec_validation(lib):
    assert upd_spec(lib, width=1) == WIDTH
    assert upd_spec(lib, sl=5) == STATE                 # shifting needs W-2+seqlen = 6 columns
    # with a buffer the line is not shifted, so W-1 columns suffice: 3 passes
    # the column check and the capacity check decides; 2 fails it
    assert upd_spec(lib, sl=3, oidx=D, oisb=4, oist=1, osteps=3) == CAP
    assert upd_spec(lib, sl=2, oidx=D, oisb=4, oist=1, osteps=4) == STATE
    assert upd_spec(lib, oidx=D, oisb=4, oist=1, osteps=3) == CAP
    assert upd_spec(lib, inter=E, isb=768, ist=192, isd=1, isw=64, isteps=3) == CAP
    assert upd_spec(lib, inter=E, isb=-1, ist=192, isd=1, isw=64, isteps=4) == STRIDE
    assert upd_spec(lib, oidx=D, oisb=-4, oist=1, osteps=4) == STRIDE
    assert upd_spec(lib, inter=B, isb=768, ist=192, isd=1, isw=64, isteps=4) == ALIAS
    assert upd_spec(lib, batch=0) == OK


def meta(lib, **over):
    args = dict(qsl=A, n_req=3, n_act=10, n_pad=16, seq=B, qs=C, cap=16, stream=None)
    args.update(over)
    return lib.paged_sconv_seq_metadata(*args.values())


def test_metadata_validation(lib):
    assert meta(lib, n_pad=9) == SIZE
    assert meta(lib, cap=15) == CAP
    assert meta(lib, n_req=0) == SIZE
    assert meta(lib, seq=None) == NULLP
    assert meta(lib, n_act=0, n_pad=0) == OK
    assert meta(lib, n_req=-1) == SIZE


def paged(lib, **over):
    args = dict(x=A, xst=2048, cache=B, csb=16 * 16 * 512, csh=16 * 512, csn=512, nb=1024, H=16,
                N=16, D=512, w=C, wsc=4, wsw=1, out=C + 65536, ost=2048, pos=C + 2 * 65536,
                sidx=C + 3 * 65536, slot=C + 4 * 65536, bt=C + 5 * 65536, btr=200, btrows=32,
                maxb=200, qs=C + 6 * 65536, T=8, off_s=128, ws=128, width=4, silu=1, resid=1,
                err=None, stream=None)
    args.update(over)
    return lib.paged_sconv_fwd(*args.values())


def test_paged_validation(lib):
    assert paged(lib, width=9) == WIDTH
    assert paged(lib, off_s=400) == RANGE  # 400 + 128 > 512
    assert paged(lib, off_s=-8) == RANGE
    assert paged(lib, H=0) == SIZE
    assert paged(lib, maxb=0) == SIZE
    assert paged(lib, csn=-512) == STRIDE
    assert paged(lib, bt=None) == NULLP
    assert paged(lib, out=A + 16) == ALIAS
    assert paged(lib, T=0) == OK


def test_binding_rejects_cpu_tensors():
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    case = wl.varlen_prefill(1, [3, 2], 16, 4)
    with pytest.raises(TypeError):
        ccv.ccv_fwd(**case.kwargs())
    d = wl.decode(2, 2, 16, 4)
    with pytest.raises(TypeError):
        ccv.ccv_update(**d.kwargs())
    p = wl.paged(3, [2], [0], H=1, ws=8, N=4, D=8, num_blocks=4, off_s=0)
    with pytest.raises(TypeError):
        ccv.paged_sconv_fwd(**p.kwargs())


def test_binding_requires_one_device_per_call():
    """Every tensor of a call must live on one device; items that are not
    tensors (the stream descriptor array) are ignored."""
    from causal_depthwise_conv1d_fwd_gb300 import api

    a, b = torch.empty(2), torch.empty(2, device="meta")
    assert api._device_of((a, None, "descs", a)) == a.device
    with pytest.raises(ValueError, match="one device"):
        api._device_of((a, b))


def test_product_path_does_not_touch_the_oracle():
    """The package must never import the oracle (no CPU fallback)."""
    import os

    from causal_depthwise_conv1d_fwd_gb300 import build as b

    pkg = os.path.dirname(b.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ccv_oracle" not in text, f


def streams_call(lib, descs, n=None, **over):
    args = dict(streams=ctypes.cast(descs, ctypes.c_void_p) if descs is not None else None,
                n=len(descs) if n is None else n, cache=B, csb=16 * 16 * 512, csh=16 * 512,
                csn=512, nb=64, H=16, N=16, D=512, pos=C, seq=D, slot=E, bt=A, btr=8, btrows=4,
                maxb=8, qs=A + 4096, T=32, width=4, silu=1, resid=1, err=None, stream=None)
    args.update(over)
    return lib.paged_sconv_fwd_streams(*args.values())


def _descs(*ranges):
    arr = (_lib.PagedStream * len(ranges))()
    for i, (off, ws) in enumerate(ranges):
        arr[i] = _lib.PagedStream(0x100000 * (i + 1), 16 * ws, 0x60000000 + 0x10000 * i, 4, 1,
                                  0x70000000 + 0x100000 * i, 16 * ws, off, ws)
    return arr


def test_paged_streams_validation(lib):
    assert streams_call(lib, _descs((0, 128), (64, 128))) == RANGE      # D-ranges overlap
    assert streams_call(lib, _descs((0, 128), (448, 128))) == RANGE     # past D
    assert streams_call(lib, _descs((0, 128)), n=0) == SIZE
    assert streams_call(lib, _descs(*[(64 * i, 64) for i in range(8)]), n=9) == SIZE
    assert streams_call(lib, None, n=2) == NULLP
    assert streams_call(lib, _descs((0, 128), (128, 128)), width=6) == WIDTH
    assert streams_call(lib, _descs((0, 128), (128, 128)), T=0) == OK


def test_missing_library_fails_loudly(tmp_path):
    """Without libccv.so the binding raises; it never falls back to another path."""
    code = (
        "import causal_depthwise_conv1d_fwd_gb300._lib as L\n"
        f"L.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "L._LIB = None\n"
        "try:\n"
        "    L.load()\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    raise SystemExit('no error')\n")
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert proc.returncode == 0, proc.stderr
    assert "not built" in proc.stdout


def test_binding_rejects_a_strided_or_misshapen_bias():
    """The C ABI reads bias as dim contiguous values, so the binding refuses a
    strided view (a column of a packed parameter) and a wrong length instead
    of passing a pointer the kernels would misread."""
    from causal_depthwise_conv1d_fwd_gb300 import api

    packed = torch.zeros(16, 3)
    assert api._bias_vector(None, 16) is None
    assert api._bias_vector(packed[:, 0].contiguous(), 16) is not None
    with pytest.raises(ValueError, match="contiguous"):
        api._bias_vector(packed[:, 1], 16)
    with pytest.raises(ValueError, match="shape"):
        api._bias_vector(torch.zeros(15), 16)
    # a single channel has no stride to get wrong
    assert api._bias_vector(packed[:1, 2], 1) is not None


def paged_meta(lib, **over):
    args = dict(x=A, xst=2048, cache=B, csb=16 * 16 * 512, csh=16 * 512, csn=512, nb=1024, H=16,
                N=16, D=512, w=C, wsc=4, wsw=1, out=C + 65536, ost=2048, pos=C + 2 * 65536,
                qsl=C + 3 * 65536, nreq=3, nact=8, seqo=None, qso=None, slot=C + 4 * 65536,
                bt=C + 5 * 65536, btr=200, btrows=32, maxb=200, T=8, off_s=128, ws=128, width=4,
                silu=1, resid=1, err=None, stream=None)
    args.update(over)
    return lib.paged_sconv_fwd_with_metadata(*args.values())


def test_paged_with_metadata_validation(lib):
    assert paged_meta(lib, nact=9) == SIZE     # more real tokens than rows
    assert paged_meta(lib, nreq=0) == SIZE     # real tokens but no request
    assert paged_meta(lib, nreq=-1) == SIZE
    assert paged_meta(lib, qsl=None) == NULLP
    assert paged_meta(lib, width=9) == WIDTH
    assert paged_meta(lib, off_s=400) == RANGE
    assert paged_meta(lib, out=A + 16) == ALIAS
    assert paged_meta(lib, bt=None) == NULLP
    assert paged_meta(lib, T=0, nact=0) == OK
