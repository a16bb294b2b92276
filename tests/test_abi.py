"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments with status codes.  No test here launches a kernel or needs a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "attn_block_mask.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"attn_block_mask_workspace_size", "attn_block_mask_build", "attn_fwd", "attn_bwd",
            "attn_get_status", "attn_status_string", "attn_version",
            "attn_last_error_message"} <= names


def test_library_exports_every_declared_symbol(native_lib):
    for name in declared_functions():
        assert hasattr(native_lib, name), name


def test_status_strings(native_lib):
    from block_sparse_masked_mask_gb300 import api
    for code in api.STATUS:
        s = api.attn_status_string(code)
        assert s and s != "unknown status"
    assert api.attn_status_string(99) == "unknown status"
    assert api.attn_version() >= 100


def test_workspace_size_is_host_only_and_validates(native_lib):
    from block_sparse_masked_mask_gb300 import api
    a = api.attn_block_mask_workspace_size(1, 32768, 32768)
    b = api.attn_block_mask_workspace_size(12, 32768, 7869)
    assert a > 0 and b > 0
    # the label matrix is NQ x NK, so a longer max_seqlen never needs less
    assert api.attn_block_mask_workspace_size(1, 4096, 4096) >= api.attn_block_mask_workspace_size(1, 4096, 1024)
    out = ctypes.c_size_t()
    lib = native_lib
    assert lib.attn_block_mask_workspace_size(1, 100, 100, 64, 128, ctypes.byref(out)) == 2
    assert lib.attn_block_mask_workspace_size(-1, 100, 100, 128, 128, ctypes.byref(out)) == 1
    assert lib.attn_block_mask_workspace_size(1, -5, 100, 128, 128, ctypes.byref(out)) == 1
    assert lib.attn_block_mask_workspace_size(1, 100, 100, 128, 128, None) == 1


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_build_rejects_bad_arguments_before_any_launch(native_lib):
    from block_sparse_masked_mask_gb300 import _native
    lib = native_lib
    out = _native.AttnBlockMask()
    prm = _native.AttnMaskParams(1)
    args = dict(kind=0, cu=_fake(), batch=1, T=256, maxL=256, seg=None, role=None, turn=None,
                bm_=128, bn=128, ws=_fake(0x20000), wsb=1 << 20)

    def call(**kw):
        a = dict(args, **kw)
        return lib.attn_block_mask_build(a["kind"], ctypes.byref(prm), a["cu"], a["batch"], a["T"],
                                         a["maxL"], a["seg"], a["role"], a["turn"], a["bm_"], a["bn"],
                                         a["ws"], a["wsb"], ctypes.byref(out), None)

    assert call(cu=None) == 1
    assert call(ws=None) == 1
    assert call(kind=7) == 1
    assert call(batch=0) == 1
    assert call(bm_=64) == 2
    assert call(kind=1) == 1            # causal_document needs seg_id
    assert call(kind=2) == 1            # shared_prefix needs seg_id
    assert call(kind=3, role=_fake()) == 1  # strip_thinking needs role and turn
    assert call(kind=4, turn=_fake()) == 1  # so does its duplicated-answer variant
    assert call(kind=6) == 1                # dense needs its bits and offsets
    assert call(ws=_fake(0x20010)) == 1   # workspace not 256-byte aligned
    assert call(wsb=16) == 3             # workspace too small


def test_dup_kind_reserves_answer_role_codes(native_lib):
    """The duplicated-answer kind takes roles 2 and 3 for the two answer
    copies, so THINK may not be either."""
    from block_sparse_masked_mask_gb300 import _native
    out = _native.AttnBlockMask()
    for rt, want in ((2, 1), (3, 1)):
        prm = _native.AttnMaskParams(rt)
        for fn in (native_lib.attn_block_mask_build, native_lib.attn_block_mask_build_noalloc):
            assert fn(4, ctypes.byref(prm), _fake(), 1, 256, 256, None, _fake(), _fake(), 128, 128,
                      _fake(0x20000), 1 << 20, ctypes.byref(out), None) == want


def test_fwd_rejects_bad_arguments_before_any_launch(native_lib):
    from block_sparse_masked_mask_gb300 import _native
    lib = native_lib
    bm = _native.AttnBlockMask()   # magic 0: never built
    prm = _native.AttnMaskParams(1)
    base = dict(q=_fake(), k=_fake(), v=_fake(), o=_fake(), lse=_fake(), dtype=0, T=256, H=2,
                D=128, scale=0.0, cu=_fake(0x30000), batch=1, maxL=256, kind=0, seg=None,
                role=None, turn=None)

    def call(bmref=bm, **kw):
        a = dict(base, **kw)
        return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dtype"], a["T"], a["H"],
                            a["D"], a["scale"], a["cu"], a["batch"], a["maxL"], a["kind"],
                            ctypes.byref(prm), a["seg"], a["role"], a["turn"],
                            ctypes.byref(bmref), None)

    assert call(q=None) == 1
    assert call(D=96) == 2
    assert call(dtype=5) == 1
    assert call(scale=-1.0) == 1
    assert call(H=0) == 1
    assert call(q=_fake(0x10008)) == 1          # q not 16-byte aligned
    assert call(kind=1) == 1                    # causal_document without seg_id
    assert call() == 4                          # block mask never built
    # a mask that claims another kind / cu_seqlens is refused
    bm2 = _native.AttnBlockMask()
    bm2.magic = 0x4B53414D
    bm2.kind, bm2.role_think, bm2.batch, bm2.total_tokens, bm2.max_seqlen = 0, 1, 1, 256, 256
    bm2.block_m = bm2.block_n = 128
    bm2.cu_seqlens = 0x30000
    assert call(bmref=bm2, kind=1, seg=_fake()) == 4
    assert call(bmref=bm2, cu=_fake(0x40000)) == 4
    assert call(bmref=bm2, T=512) == 4


def test_bwd_rejects_bad_arguments_before_any_launch(native_lib):
    from block_sparse_masked_mask_gb300 import _native
    lib = native_lib
    bm = _native.AttnBlockMask()   # magic 0: never built
    prm = _native.AttnMaskParams(1)
    base = dict(q=_fake(), k=_fake(), v=_fake(), o=_fake(), do=_fake(), lse=_fake(),
                dq=_fake(0x60000), dk=_fake(0x70000), dv=_fake(0x80000), dtype=0, T=256, H=2,
                D=128, scale=0.0, cu=_fake(0x30000), batch=1, maxL=256, kind=0, seg=None,
                role=None, turn=None, ws=_fake(0x90000), wsb=1 << 30)

    def call(bmref=bm, **kw):
        a = dict(base, **kw)
        return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                            a["dv"], a["dtype"], a["T"], a["H"], a["D"], a["scale"], a["cu"],
                            a["batch"], a["maxL"], a["kind"], ctypes.byref(prm), a["seg"],
                            a["role"], a["turn"], ctypes.byref(bmref), a["ws"], a["wsb"], None)

    for name in ("q", "do", "lse", "dq", "dk", "dv", "ws"):
        assert call(**{name: None}) == 1, name
    assert call(dtype=1) == 2                   # fp32 backward is not provided
    assert call(dtype=5) == 1
    assert call(D=96) == 2
    assert call(scale=float("nan")) == 1
    assert call(dk=_fake(0x70008)) == 1         # dk not 16-byte aligned
    assert call(ws=_fake(0x90010)) == 1         # workspace not 256-byte aligned
    assert call(kind=3, role=_fake()) == 1      # strip_thinking without turn
    assert call() == 4                          # block mask never built
    bm2 = _native.AttnBlockMask()
    bm2.magic = 0x4B53414D
    bm2.kind, bm2.role_think, bm2.batch, bm2.total_tokens, bm2.max_seqlen = 0, 1, 1, 256, 256
    bm2.block_m = bm2.block_n = 128
    bm2.cu_seqlens = 0x30000
    assert call(bmref=bm2, maxL=128) == 4
    # workspace size: the side values of each q-tile and head (3 x 128 fp32),
    # ||dO_i|| [H, T] fp32, the bound words [batch][H][4] fp32 and the dQ
    # accumulator [T, H, D] int32, each 256-byte aligned; nothing per tile pair
    bm2.max_qtiles = 3
    out = ctypes.c_size_t()
    a256 = lambda x: (x + 255) // 256 * 256
    for kind in (0, 5):
        bm2.kind = kind
        for H, D in ((2, 128), (1, 64), (3, 32)):
            assert lib.attn_bwd_workspace_size(ctypes.byref(bm2), H, D, ctypes.byref(out)) == 0
            want = a256(4 * H * 3 * 384) + a256(4 * H * 256) + a256(16 * H) + a256(4 * 256 * H * D)
            assert out.value == want, (kind, H, D)
    bm2.kind = 0
    assert lib.attn_bwd_workspace_size(ctypes.byref(bm2), 2, 128, ctypes.byref(out)) == 0
    assert call(bmref=bm2, wsb=out.value - 1) == 3
    assert lib.attn_bwd_workspace_size(ctypes.byref(bm2), 2, 96, ctypes.byref(out)) == 2
    assert lib.attn_bwd_workspace_size(ctypes.byref(bm2), 0, 128, ctypes.byref(out)) == 1
    assert lib.attn_bwd_workspace_size(None, 2, 128, ctypes.byref(out)) == 1


def test_get_status_rejects_unbuilt_mask(native_lib):
    from block_sparse_masked_mask_gb300 import _native
    bm = _native.AttnBlockMask()
    assert native_lib.attn_get_status(ctypes.byref(bm), None) == 1
    assert native_lib.attn_get_status(None, None) == 1


def test_product_path_has_no_oracle_or_fallback():
    """The library package never imports the oracle and has no CPU fallback."""
    pkg = os.path.join(ROOT, "block_sparse_masked_mask_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), fn
    native = open(os.path.join(pkg, "_native.py")).read()
    assert "raise RuntimeError" in native


def test_binding_refuses_host_tensors_before_any_call():
    """A host tensor's pointer must never reach a kernel: the binding refuses
    it (ATTN_ERR_INVALID_ARG) before calling into the library."""
    import torch
    from block_sparse_masked_mask_gb300 import api
    q = torch.zeros((256, 2, 64), dtype=torch.bfloat16)
    lse = torch.zeros((2, 256))
    cu = torch.tensor([0, 256], dtype=torch.int32)
    for call in (lambda: api.attn_block_mask_build("causal", cu, 256, 256),
                 lambda: api.attn_fwd(q, q, q, None, "causal", cu, 256),
                 lambda: api.attn_bwd(q, q, q, q, lse, q, None, "causal", cu, 256)):
        with pytest.raises(api.AttnError) as e:
            call()
        assert e.value.status == 1 and "CUDA tensor" in str(e.value)
