"""The C-ABI library loads, exports every function include/libmla.h declares,
and its host-side validation rejects bad arguments (CPU only: none of these
calls reaches a kernel)."""
import ctypes

import pytest

import __graft_entry__ as G


@pytest.fixture(scope="module")
def lib():
    G._load_by_path("_libmla_build", "paged_mla_decode_10_gb300/build.py").build()
    from paged_mla_decode_10_gb300 import _lib
    return _lib.load()


def test_exports_every_declared_function(lib):
    from paged_mla_decode_10_gb300 import _lib
    names = _lib.header_functions()
    assert {"mla_get_metadata", "mla_decode_fwd", "mla_workspace_size", "mla_get_num_sm_parts",
            "mla_check_device_error"} <= set(names)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(7):
        assert lib.mla_status_string(code)
    assert lib.mla_version() >= 100


def _shape(**kw):
    from paged_mla_decode_10_gb300._lib import MlaShape
    sh = MlaShape()
    vals = dict(batch=2, s_q=1, h_q=16, h_k=1, head_dim=576, head_dim_v=512, page_block_size=64,
                num_blocks=8, max_blocks_per_seq=5, num_sm_parts=4)
    vals.update(kw)
    for k, v in vals.items():
        setattr(sh, k, v)
    qs = kw.get("q_stride", (16 * 576, 16 * 576, 576))
    ks = kw.get("k_stride", (64 * 576, 576, 576))
    os_ = kw.get("out_stride", (16 * 512, 16 * 512, 512))
    for i in range(3):
        sh.q_stride[i], sh.k_stride[i], sh.out_stride[i] = qs[i], ks[i], os_[i]
    sh.bt_stride = kw.get("bt_stride", 5)
    return sh


def test_workspace_size_formula(lib):
    n = ctypes.c_size_t(0)
    sh = _shape()
    assert lib.mla_workspace_size(ctypes.byref(sh), ctypes.byref(n)) == 0
    slots, rows = 2 + 4, 16
    o = slots * rows * 512 * 4
    o = (o + 255) // 256 * 256
    l = (slots * rows * 4 + 255) // 256 * 256
    assert n.value == o + l


@pytest.mark.parametrize("bad", [
    dict(head_dim=512), dict(head_dim_v=256), dict(page_block_size=32), dict(h_q=12, h_k=8),
    dict(s_q=0), dict(num_sm_parts=0), dict(num_blocks=0), dict(q_stride=(16 * 576, 16 * 576, 577)),
    dict(bt_stride=4), dict(batch=-1),
])
def test_workspace_size_rejects_bad_shapes(lib, bad):
    n = ctypes.c_size_t(0)
    sh = _shape(**bad)
    assert lib.mla_workspace_size(ctypes.byref(sh), ctypes.byref(n)) == 1   # MLA_ERR_ARG
    assert lib.mla_last_error()


def test_too_many_rows_is_unsupported(lib):
    n = ctypes.c_size_t(0)
    sh = _shape(s_q=16, h_q=128)
    assert lib.mla_workspace_size(ctypes.byref(sh), ctypes.byref(n)) == 2   # MLA_ERR_UNSUPPORTED


def test_decode_rejects_null_pointers_before_any_cuda_call(lib):
    sh = _shape()
    rc = lib.mla_decode_fwd(ctypes.byref(sh), None, None, None, None, None, None, ctypes.c_float(0.0), 0,
                            None, None, None, 0, None)
    assert rc == 1


def test_metadata_rejects_bad_arguments(lib):
    assert lib.mla_get_metadata(None, 4, 128, 1, 76, None, None, None) == 1
    dummy = ctypes.c_void_p(256)
    assert lib.mla_get_metadata(dummy, -1, 128, 1, 76, dummy, dummy, None) == 1
    assert lib.mla_get_metadata(dummy, 4, 128, 1, 0, dummy, dummy, None) == 1
    # the one-byte / two-byte cache variant: any other element size is an argument error
    assert lib.mla_get_metadata_ex(dummy, 4, 128, 1, 3, 76, dummy, dummy, None) == 1
    assert lib.mla_get_metadata_ex(None, 4, 128, 1, 1, 76, None, None, None) == 1


def test_host_decode_rejects_bad_arguments_before_any_cuda_call(lib):
    dummy = ctypes.c_void_p(256)
    sh = _shape()
    args = lambda s, q=dummy, out=dummy: (ctypes.byref(s), q, dummy, dummy, dummy, ctypes.c_float(0.0), 0, out,
                                          dummy, None)
    assert lib.mla_decode_fwd_host(*args(sh, q=None)) == 1                                # NULL q
    assert lib.mla_decode_fwd_host(*args(sh, out=ctypes.c_void_p(264))) == 1              # out not 16-byte aligned
    assert lib.mla_decode_fwd_host(*args(_shape(out_stride=(32 * 512, 16 * 512, 512)))) == 1   # out not contiguous
    assert b"contiguous" in lib.mla_last_error()
    assert lib.mla_decode_fwd_host(*args(_shape(num_sm_parts=1025))) == 2                 # schedule limit
    assert lib.mla_decode_fwd_host(*args(_shape(head_dim=512))) == 1                      # bad shape


def test_split_decode_rejects_bad_arguments_before_any_cuda_call(lib):
    from paged_mla_decode_10_gb300._lib import MlaRopeStrides
    dummy = ctypes.c_void_p(256)
    sh = _shape(q_stride=(16 * 512, 16 * 512, 512), k_stride=(64 * 512, 512, 512))
    rs = MlaRopeStrides()
    for i, (a, b) in enumerate(zip((16 * 64, 16 * 64, 64), (64 * 64, 64, 64))):
        rs.q_rope_stride[i], rs.krope_stride[i] = a, b

    def call(rope=ctypes.byref(rs), q_rope=dummy, krope=dummy, shape=sh):
        return lib.mla_decode_fwd_split(ctypes.byref(shape), rope, dummy, q_rope, dummy, krope, dummy, dummy, dummy,
                                        dummy, ctypes.c_float(0.0), 0, dummy, dummy, dummy, 1 << 30, None)
    assert call(rope=None) == 1                              # no rope strides
    assert call(q_rope=None) == 1                            # NULL q_rope
    assert call(krope=ctypes.c_void_p(264)) == 1             # krope not 16-byte aligned
    rs.krope_stride[2] = 60
    assert call() == 1                                       # stride not a multiple of 8
    rs.krope_stride[2] = 56
    assert call() == 1                                       # head stride below 64 dims
    rs.krope_stride[2] = 64
    assert call(shape=_shape(q_stride=(16 * 512, 16 * 512, 504), k_stride=(64 * 512, 512, 512))) == 1


def test_fp8_decode_rejects_bad_arguments_before_any_cuda_call(lib):
    dummy = ctypes.c_void_p(256)

    def call(shape=None, q=dummy, bmm1=0.04, bmm2=1.0, fn="mla_decode_fwd_fp8"):
        sh = shape or _shape()
        return getattr(lib, fn)(ctypes.byref(sh), q, dummy, dummy, dummy, dummy, dummy, ctypes.c_float(bmm1),
                                ctypes.c_float(bmm2), 0, dummy, dummy, dummy, 1 << 30, None)
    for fn in ("mla_decode_fwd_fp8", "mla_decode_splitkv_fp8"):
        assert call(q=None, fn=fn) == 1                                   # NULL q
        assert call(q=ctypes.c_void_p(264), fn=fn) == 1                   # q not 16-byte aligned
        for bad in (0.0, -1.0, float("nan"), float("inf")):
            assert call(bmm1=bad, fn=fn) == 1                             # bmm1_scale not positive and finite
        assert b"bmm1_scale" in lib.mla_last_error()
        assert call(bmm2=float("nan"), fn=fn) == 1                        # bmm2_scale not finite
        # a head stride of 584 bytes: a multiple of 8 elements but not of 16 bytes
        assert call(shape=_shape(q_stride=(16 * 584, 16 * 584, 584)), fn=fn) == 1
        assert b"16" in lib.mla_last_error()
        assert call(shape=_shape(head_dim=512), fn=fn) == 1              # bad shape
