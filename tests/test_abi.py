"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, sizes its workspace, and rejects bad arguments before any
device work. No kernel runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "saf.h")


@pytest.fixture(scope="module")
def saf():
    from softmax_attention_hybrid_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from softmax_attention_hybrid_gb300 import saf as mod
    return mod


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(saf_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    assert {"saf_attn_fwd", "saf_attn_bwd", "saf_attn_workspace_bytes", "saf_device_status",
            "saf_error_string"} <= set(names)


def test_library_exports_every_declared_symbol(saf):
    lib = saf.library()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(saf.EXPORTED)


def test_version_and_error_strings(saf):
    assert saf.saf_version() >= 100
    for st in (0, -1, -2, -3, -4, -5, -6, -8, -99):
        s = saf.saf_error_string(st)
        assert isinstance(s, str) and s


def test_workspace_bytes(saf):
    f = saf.saf_attn_workspace_bytes
    assert f(8, 12, 4096, 64, "bf16", 0) > 0
    assert f(8, 12, 4096, 64, "bf16", 1) > f(8, 12, 4096, 64, "bf16", 0)
    assert f(8, 12, 4096, 64, "bf16", 1) % 256 == 0
    assert f(1, 4, 256, 32, "bf16", 0) == 0        # unsupported d
    assert f(1, 4, 256, 80, "bf16", 0) == 0        # unsupported d
    assert f(1, 4, 256, 96, "bf16", 1) > 0 and f(1, 4, 256, 128, "bf16", 0) > 0
    assert f(1, 4, 256, 96, "fp32", 1) > 0 and f(1, 4, 256, 128, "fp32", 0) > 0
    assert f(1, 0, 256, 64, "bf16", 0) == 0        # no heads
    assert f(1, 300, 256, 64, "bf16", 0) == 0      # more than SAF_MAX_HEADS
    assert f(0, 4, 0, 64, "fp32", 1) > 0           # empty call still has the status words


FAKE = 0x10000  # 64 KiB-aligned fake device address: the calls below must fail before any access


def _fwd(lib, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, a=FAKE, r=FAKE, ld=256, frozen=None, B=1, H=4, T=256, d=64, dt=0,
                o=FAKE, lse=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    fz = args["frozen"]
    fzp = (ctypes.c_uint8 * len(fz))(*fz) if fz is not None else None
    return lib.saf_attn_fwd(args["q"], args["k"], args["v"], args["a"], args["r"], args["ld"], fzp, args["B"],
                            args["H"], args["T"], args["d"], args["dt"], args["o"], args["lse"], args["ws"],
                            args["wsb"], args["stream"])


def test_argument_errors_return_before_device_work(saf):
    lib = saf.library()
    assert _fwd(lib, H=0) == saf.SAF_EINVAL
    assert _fwd(lib, B=-1) == saf.SAF_EINVAL
    assert _fwd(lib, H=257, frozen=None) == saf.SAF_EINVAL
    assert _fwd(lib, d=80) == saf.SAF_EUNSUPPORTED
    assert _fwd(lib, dt=7) == saf.SAF_EINVAL
    assert _fwd(lib, v=None) == saf.SAF_EINVAL
    assert _fwd(lib, q=None) == saf.SAF_EINVAL                           # ordinary heads need q
    assert _fwd(lib, frozen=[1, 1, 1, 1], q=None, k=None, ws=None) == saf.SAF_EWORKSPACE  # q, k unused
    assert _fwd(lib, frozen=[0, 1, 0, 0], a=None) == saf.SAF_EINVAL      # frozen heads need a, r
    assert _fwd(lib, frozen=[0, 1, 0, 0], ld=255) == saf.SAF_EINVAL      # ld_prior < T
    assert _fwd(lib, v=FAKE + 8) == saf.SAF_EALIGN
    assert _fwd(lib, ws=FAKE + 16) == saf.SAF_EALIGN
    assert _fwd(lib, ws=None) == saf.SAF_EWORKSPACE
    assert _fwd(lib, wsb=16) == saf.SAF_EWORKSPACE


def test_empty_call_is_a_no_op(saf):
    lib = saf.library()
    assert _fwd(lib, T=0, q=None, k=None, v=None, o=None, lse=None, ws=None) == saf.SAF_OK
    assert _fwd(lib, B=0, q=None, k=None, v=None, o=None, lse=None, ws=None) == saf.SAF_OK


def test_bwd_argument_errors(saf):
    lib = saf.library()
    F = FAKE

    def bwd(**kw):
        a = dict(q=F, k=F, v=F, o=F, do=F, lse=F, a=F, r=F, ld=256, B=1, H=4, T=256, d=64, dt=0,
                 dq=F, dk=F, dv=F, ws=F, wsb=1 << 30)
        a.update(kw)
        return lib.saf_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["a"], a["r"], a["ld"],
                                None, a["B"], a["H"], a["T"], a["d"], a["dt"], a["dq"], a["dk"], a["dv"],
                                a["ws"], a["wsb"], None)

    assert bwd(dq=None) == saf.SAF_EINVAL
    assert bwd(do=F + 4) == saf.SAF_EALIGN
    assert bwd(wsb=1024) == saf.SAF_EWORKSPACE
    assert bwd(T=0) == saf.SAF_OK
    assert bwd(d=80) == saf.SAF_EUNSUPPORTED


def test_device_status_rejects_null(saf):
    assert saf.library().saf_device_status(None, None) == saf.SAF_EWORKSPACE


def test_no_device_is_reported_not_faked(saf):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # every argument valid: the call reaches the device check and must fail there
    assert _fwd(saf.library()) in (saf.SAF_ECUDA, saf.SAF_EUNSUPPORTED)


def test_fit_argument_errors(saf):
    lib = saf.library()
    F = FAKE
    assert saf.saf_fit_workspace_bytes(3, 4096) > 0 and saf.saf_fit_workspace_bytes(3, 4096) % 256 == 0
    assert saf.saf_fit_workspace_bytes(0, 16) == 0 and saf.saf_fit_workspace_bytes(2, 0) == 0

    def fit(**kw):
        a = dict(ea=F, er=F, H=2, T=64, steps=400, lr=0.05, a=F, r=F, loss=F, ws=F, wsb=1 << 30)
        a.update(kw)
        return lib.saf_fit_compact(a["ea"], a["er"], a["H"], a["T"], a["steps"], a["lr"], a["a"], a["r"],
                                   a["loss"], a["ws"], a["wsb"], None)

    assert fit(H=0) == saf.SAF_EINVAL
    assert fit(T=0) == saf.SAF_EINVAL
    assert fit(steps=-1) == saf.SAF_EINVAL
    assert fit(lr=0.0) == saf.SAF_EINVAL
    assert fit(lr=float("nan")) == saf.SAF_EINVAL
    assert fit(ea=None) == saf.SAF_EINVAL
    assert fit(a=F + 2) == saf.SAF_EALIGN
    assert fit(ws=None) == saf.SAF_EWORKSPACE
    assert fit(ws=F + 64) == saf.SAF_EALIGN
    assert fit(wsb=256) == saf.SAF_EWORKSPACE


def test_pattern_grad_argument_errors(saf):
    lib = saf.library()
    F = FAKE

    def pg(**kw):
        a = dict(v=F, do=F, o=F, lse=F, a=F, r=F, ld=256, B=1, H=4, T=256, d=64, dt=0, da=F, dr=F, frozen=None)
        a.update(kw)
        fz = a["frozen"]
        fzp = (ctypes.c_uint8 * len(fz))(*fz) if fz is not None else None
        return lib.saf_pattern_grad(a["v"], a["do"], a["o"], a["lse"], a["a"], a["r"], a["ld"], fzp, a["B"],
                                    a["H"], a["T"], a["d"], a["dt"], a["da"], a["dr"], None)

    assert pg(H=0) == saf.SAF_EINVAL
    assert pg(d=80) == saf.SAF_EUNSUPPORTED
    assert pg(d=96, da=None) == saf.SAF_EINVAL   # d = 96 and 128 are served: the next check answers
    assert pg(dt=5) == saf.SAF_EINVAL
    assert pg(da=None) == saf.SAF_EINVAL
    assert pg(dr=F + 1) == saf.SAF_EALIGN
    assert pg(T=0) == saf.SAF_OK
    # with a frozen head there is work to do: the remaining arguments are checked
    # before anything is enqueued (da and dr are cleared on the stream only after
    # every check), so these return their own error, not a device error
    fz = [0, 1, 0, 0]
    assert pg(frozen=fz, v=None) == saf.SAF_EINVAL
    assert pg(frozen=fz, ld=255) == saf.SAF_EINVAL
    assert pg(frozen=fz, lse=F + 4) == saf.SAF_EALIGN
    assert pg(frozen=fz, a=F + 2) == saf.SAF_EALIGN


def test_pattern_grad_tc_argument_errors(saf):
    lib = saf.library()
    F = FAKE
    need = lib.saf_pattern_grad_tc_workspace_bytes(2, 4, 256, 1)
    assert need > 0
    # the workspace grows with the batch and the number of frozen heads
    assert lib.saf_pattern_grad_tc_workspace_bytes(2, 4, 256, 2) > need
    assert lib.saf_pattern_grad_tc_workspace_bytes(4, 4, 256, 1) > need
    for bad in ((-1, 4, 256, 1), (2, 0, 256, 0), (2, 4, -1, 1), (2, 4, 256, 5), (2, 4, 256, -1)):
        assert lib.saf_pattern_grad_tc_workspace_bytes(*bad) == 0, bad

    def pg(**kw):
        a = dict(v=F, do=F, o=F, lse=F, a=F, r=F, ld=256, B=2, H=4, T=256, d=64, da=F, dr=F, frozen=None,
                 ws=F, wsb=need)
        a.update(kw)
        fz = a["frozen"]
        fzp = (ctypes.c_uint8 * len(fz))(*fz) if fz is not None else None
        return lib.saf_pattern_grad_tc(a["v"], a["do"], a["o"], a["lse"], a["a"], a["r"], a["ld"], fzp, a["B"],
                                       a["H"], a["T"], a["d"], a["da"], a["dr"], a["ws"], a["wsb"], None)

    assert pg(H=0) == saf.SAF_EINVAL
    assert pg(B=-1) == saf.SAF_EINVAL
    assert pg(d=80) == saf.SAF_EUNSUPPORTED
    assert pg(d=128, da=None) == saf.SAF_EINVAL   # d = 96 and 128 are served: the next check answers
    assert pg(da=None) == saf.SAF_EINVAL
    assert pg(dr=F + 1) == saf.SAF_EALIGN
    assert pg(T=0) == saf.SAF_OK
    # with a frozen head, every argument and the workspace are checked before any work
    fz = [0, 1, 0, 0]
    assert pg(frozen=fz, v=None) == saf.SAF_EINVAL
    assert pg(frozen=fz, ld=255) == saf.SAF_EINVAL
    assert pg(frozen=fz, o=F + 8) == saf.SAF_EALIGN
    assert pg(frozen=fz, r=F + 2) == saf.SAF_EALIGN
    assert pg(frozen=fz, ws=None) == saf.SAF_EWORKSPACE
    assert pg(frozen=fz, ws=F + 128) == saf.SAF_EALIGN
    assert pg(frozen=fz, wsb=need - 1) == saf.SAF_EWORKSPACE


def test_gqa_argument_errors(saf):
    lib = saf.library()
    F = FAKE

    def fwd(**kw):
        a = dict(H=8, Hkv=2, frozen=None, T=256, ws=F)
        a.update(kw)
        fz = a["frozen"]
        fzp = (ctypes.c_uint8 * len(fz))(*fz) if fz is not None else None
        return lib.saf_attn_fwd_gqa(F, F, F, F, F, 256, fzp, 1, a["H"], a["Hkv"], a["T"], 64, 0, F, F, a["ws"],
                                    1 << 30, None)

    def bwd(**kw):
        a = dict(H=8, Hkv=2, T=256, d=64)
        a.update(kw)
        return lib.saf_attn_bwd_gqa(F, F, F, F, F, F, F, F, 256, None, 1, a["H"], a["Hkv"], a["T"], a["d"], 0, F, F,
                                    F, F, 1 << 30, None)

    assert fwd(Hkv=0) == saf.SAF_EINVAL
    assert fwd(Hkv=3) == saf.SAF_EINVAL           # 8 query heads do not split over 3
    assert fwd(Hkv=16) == saf.SAF_EINVAL          # more key/value heads than query heads
    assert fwd(ws=None) == saf.SAF_EWORKSPACE     # a valid layout reaches the later checks
    assert fwd(T=0, ws=None) == saf.SAF_OK
    assert bwd(Hkv=-1) == saf.SAF_EINVAL
    assert bwd(Hkv=5) == saf.SAF_EINVAL
    assert bwd(T=0) == saf.SAF_OK
    # bf16 at d = 96 / 128 serves the grouped layout too: these calls get past the head
    # dimension and stop at the missing output (o, dq = NULL), before any device work
    assert lib.saf_attn_bwd_gqa(F, F, F, F, F, F, F, F, 256, None, 1, 8, 2, 256, 128, 0, None, F, F, F, 1 << 30,
                                None) == saf.SAF_EINVAL
    assert lib.saf_attn_fwd_gqa(F, F, F, F, F, 256, None, 1, 8, 2, 256, 96, 0, None, F, F, 1 << 30,
                                None) == saf.SAF_EINVAL
    assert lib.saf_attn_fwd_gqa(F, F, F, F, F, 256, None, 1, 8, 2, 256, 80, 0, None, F, F, 1 << 30,
                                None) == saf.SAF_EUNSUPPORTED


def test_fit_target_argument_errors(saf):
    lib = saf.library()
    F = FAKE
    assert lib.saf_fit_stats_workspace_bytes(3, 256) > 0 and lib.saf_fit_stats_workspace_bytes(0, 256) == 0
    assert lib.saf_fit_from_target_workspace_bytes(3, 256) >= lib.saf_fit_workspace_bytes(3, 256)

    def stats(**kw):
        a = dict(A=F, H=3, T=64, ea=F, er=F, ng=F, ws=F, wsb=1 << 30)
        a.update(kw)
        return lib.saf_fit_target_stats(a["A"], a["H"], a["T"], a["ea"], a["er"], a["ng"], a["ws"], a["wsb"], None)

    def pipe(**kw):
        a = dict(A=F, H=3, T=64, steps=400, lr=0.05, tol=0.2, a=F, r=F, k=F, acc=F, ws=F, wsb=1 << 30)
        a.update(kw)
        return lib.saf_fit_from_target(a["A"], a["H"], a["T"], a["steps"], a["lr"], a["tol"], a["a"], a["r"],
                                       a["k"], a["acc"], a["ws"], a["wsb"], None)

    assert stats(H=0) == saf.SAF_EINVAL
    assert stats(A=None) == saf.SAF_EINVAL
    assert stats(ea=F + 2) == saf.SAF_EALIGN
    assert stats(ws=None) == saf.SAF_EWORKSPACE
    assert stats(wsb=16) == saf.SAF_EWORKSPACE
    assert pipe(steps=-1) == saf.SAF_EINVAL
    assert pipe(tol=-0.1) == saf.SAF_EINVAL
    assert pipe(lr=0.0) == saf.SAF_EINVAL
    assert pipe(acc=None) == saf.SAF_EINVAL
    assert pipe(k=F + 1) == saf.SAF_EALIGN
    assert pipe(ws=F + 128) == saf.SAF_EALIGN
    assert pipe(wsb=4096) == saf.SAF_EWORKSPACE


def test_diag_argument_errors(saf):
    lib = saf.library()
    F = FAKE

    def diag(**kw):
        a = dict(dt=0, withhold=1, wait=1000, ws=F)
        a.update(kw)
        return lib.saf_attn_fwd_diag(F, F, F, F, F, 256, None, 1, 4, 256, 64, a["dt"], F, F, a["ws"], 1 << 30,
                                     None, a["withhold"], a["wait"])

    assert diag(dt=1) == saf.SAF_EUNSUPPORTED     # the test switches live in the d = 64 tensor-core forward
    assert diag(withhold=2) == saf.SAF_EINVAL
    assert diag(ws=None) == saf.SAF_EWORKSPACE


def test_prepared_state_argument_errors(saf):
    lib = saf.library()
    F = FAKE
    assert lib.saf_frozen_state_bytes(4, 256, 0) > lib.saf_frozen_state_bytes(4, 256, 1) > 0
    assert lib.saf_frozen_state_bytes(0, 256, 0) == 0 and lib.saf_frozen_state_bytes(4, 256, 7) == 0
    fz = (ctypes.c_uint8 * 4)(0, 1, 0, 0)
    prep = lambda **kw: lib.saf_frozen_prepare(kw.get("a", F), F, kw.get("ld", 256), fz, 4, 256, 0,
                                               kw.get("st", F), kw.get("sb", 1 << 30), None)
    assert prep(a=None) == saf.SAF_EINVAL
    assert prep(ld=100) == saf.SAF_EINVAL
    assert prep(st=None) == saf.SAF_EWORKSPACE
    assert prep(st=F + 64) == saf.SAF_EALIGN
    assert prep(sb=1024) == saf.SAF_EWORKSPACE
    fwd = lambda **kw: lib.saf_attn_fwd_prepared(F, F, F, F, F, 256, fz, kw.get("st", F), 1, 4, kw.get("hkv", 4),
                                                 256, 64, 0, F, F, F, 1 << 30, None)
    assert fwd(st=None) == saf.SAF_EWORKSPACE
    assert fwd(hkv=3) == saf.SAF_EINVAL
    # the prepared calls take d = 96 and 128 in bf16 too (these stop at o = NULL), not 80
    assert lib.saf_attn_fwd_prepared(F, F, F, F, F, 256, fz, F, 1, 4, 4, 256, 128, 0, None, F, F, 1 << 30,
                                     None) == saf.SAF_EINVAL
    assert lib.saf_attn_fwd_prepared(F, F, F, F, F, 256, fz, F, 1, 4, 4, 256, 80, 0, None, F, F, 1 << 30,
                                     None) == saf.SAF_EUNSUPPORTED
