"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/gdn.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from gated_deltanet_wise_b300 import build
    build.build()
    from gated_deltanet_wise_b300 import gdn
    return gdn.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    from gated_deltanet_wise_b300 import gdn
    assert sorted(gdn.EXPORTED) == names


def test_version_and_status_strings(L):
    from gated_deltanet_wise_b300 import gdn
    assert L.gdn_version() >= 100
    for s in range(6):
        assert gdn.status_string(s)
    assert gdn.status_string(99) == "unknown status"


def test_workspace_sizes(L):
    from gated_deltanet_wise_b300 import gdn
    SZ_ERR = 2 ** 64 - 1
    assert gdn.gdn_frame_fwd_workspace_size(1, 20, 121, 880, 112) > 20 * 121 * 80000
    assert gdn.gdn_frame_fwd_workspace_size(1, 20, 0, 880, 112) == 0
    assert gdn.gdn_frame_fwd_workspace_size(0, 20, 4, 880, 112) == 0
    assert gdn.gdn_frame_fwd_workspace_size(1, 20, 4, 0, 112) == 0
    assert gdn.gdn_frame_fwd_workspace_size(-1, 20, 4, 8, 112) == SZ_ERR
    assert gdn.gdn_frame_fwd_workspace_size(1, 1, 4, 8, 64) == SZ_ERR   # bf16 path is D = 112
    assert gdn.gdn_frame_step_workspace_size(1, 20, 880, 112) == 0   # the fused step needs no scratch
    assert gdn.gdn_frame_step_workspace_size(1, 20, 880, 64) == 2 ** 64 - 1
    # the options entry: the sum reading matches gdn_frame_fwd, unknown flags are refused
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, 0) == \
        gdn.gdn_frame_fwd_workspace_size(1, 20, 121, 880, 112)
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, gdn.GDN_FWD_REVERSE) == \
        gdn.gdn_frame_fwd_workspace_size(1, 20, 121, 880, 112)
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, gdn.GDN_FWD_PRODUCT) == \
        gdn.gdn_frame_fwd_product_workspace_size(1, 20, 121, 880, 112)
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, gdn.GDN_FWD_FUSED) == \
        gdn.gdn_frame_fwd_workspace_size(1, 20, 121, 880, 112)
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, gdn.GDN_FWD_FUSED | gdn.GDN_FWD_PRODUCT) == \
        SZ_ERR
    assert gdn.gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, 8) == SZ_ERR
    # the workspace grows linearly in frames (per-frame images dominate)
    a = gdn.gdn_frame_fwd_workspace_size(1, 4, 10, 880, 112)
    b = gdn.gdn_frame_fwd_workspace_size(1, 4, 20, 880, 112)
    assert 1.8 < b / a < 2.2


def test_host_side_validation_without_gpu(L):
    from gated_deltanet_wise_b300 import gdn
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    args = dict(q=fake, k=fake, v=fake, beta=fake, gamma=fake, S_in=None, S_out=fake, o=fake)

    def fwd(B, H, F, N, D, ws=None, nbytes=0, **over):
        a = dict(args, **over)
        return L.gdn_frame_fwd(a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["S_in"], a["S_out"], a["o"],
                               B, H, F, N, D, 0.0, ws, nbytes, None)

    assert fwd(-1, 1, 1, 1, 112) == gdn.GDN_ERR_INVALID_ARG
    assert fwd(1, 1, 1, 1, 0) == gdn.GDN_ERR_INVALID_ARG
    assert fwd(0, 4, 4, 4, 112) == gdn.GDN_OK            # empty batch: no-op
    assert fwd(1, 1, 2, 8, 64) == gdn.GDN_ERR_UNSUPPORTED
    assert fwd(1, 1, 2, 8, 112, q=None) == gdn.GDN_ERR_INVALID_ARG
    assert fwd(1, 1, 2, 8, 112, k=P(0x10008)) == gdn.GDN_ERR_INVALID_ARG   # misaligned
    assert fwd(1, 1, 2, 8, 112, S_out=P(0x10004)) == gdn.GDN_ERR_INVALID_ARG
    assert fwd(1, 1, 2, 8, 112, ws=None, nbytes=0) == gdn.GDN_ERR_WORKSPACE
    need = gdn.gdn_frame_fwd_workspace_size(1, 1, 2, 8, 112)
    assert fwd(1, 1, 2, 8, 112, ws=fake, nbytes=need - 16) == gdn.GDN_ERR_WORKSPACE
    a = args
    for flags in (8, 16, 0x80000000):
        assert L.gdn_frame_fwd_ex(a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["S_in"], a["S_out"], a["o"],
                                  1, 1, 2, 8, 112, 0.0, flags, fake, need, None) == gdn.GDN_ERR_INVALID_ARG
    # the fused chained scan is the sum reading only
    assert L.gdn_frame_fwd_ex(a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["S_in"], a["S_out"], a["o"],
                              1, 1, 2, 8, 112, 0.0, gdn.GDN_FWD_FUSED | gdn.GDN_FWD_PRODUCT, fake, need,
                              None) == gdn.GDN_ERR_UNSUPPORTED
    assert fwd(1, 1, 2, 8, 112, ws=P(0x10008), nbytes=need) == gdn.GDN_ERR_INVALID_ARG
    def step(B, H, N, D, **over):
        a = dict(args, **over)
        return L.gdn_frame_step(a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["S_in"], a["S_out"], a["o"],
                                B, H, N, D, 0.0, None, 0, None)

    assert step(1, 1, 8, -3) == gdn.GDN_ERR_INVALID_ARG
    assert step(1, -1, 8, 112) == gdn.GDN_ERR_INVALID_ARG
    assert step(0, 20, 880, 112) == gdn.GDN_OK           # empty batch: no-op
    assert step(1, 1, 8, 128) == gdn.GDN_ERR_UNSUPPORTED
    assert step(1, 1, 8, 112, v=None) == gdn.GDN_ERR_INVALID_ARG
    assert step(1, 1, 8, 112, gamma=None) == gdn.GDN_ERR_INVALID_ARG
    assert step(1, 1, 8, 112, o=P(0x10002)) == gdn.GDN_ERR_INVALID_ARG   # misaligned
    assert step(1, 1, 8, 112, S_in=P(0x10004)) == gdn.GDN_ERR_INVALID_ARG
    comp = L.gdn_frame_composite
    assert comp(fake, fake, fake, fake, fake, fake, 1, 1, 2, 8, 64, 0.0, None, 0, None) == gdn.GDN_ERR_UNSUPPORTED
    assert comp(fake, fake, fake, None, fake, fake, 1, 1, 2, 8, 112, 0.0, None, 0, None) == gdn.GDN_ERR_INVALID_ARG
    assert comp(fake, fake, fake, fake, fake, fake, 1, 1, 2, 8, 112, 0.0, None, 0, None) == gdn.GDN_ERR_WORKSPACE
    assert comp(fake, fake, fake, fake, P(0x10004), fake, 1, 1, 2, 8, 112, 0.0, None, 0, None) == gdn.GDN_ERR_INVALID_ARG
    # no composites wanted (the last rank of a frame split): the null outputs pass validation,
    # and the call goes on to the workspace check like any other
    assert comp(fake, fake, fake, fake, None, None, 1, 1, 2, 8, 112, 0.0, None, 0, None) == gdn.GDN_ERR_WORKSPACE
    assert comp(fake, fake, fake, fake, None, P(0x10004), 1, 1, 2, 8, 112, 0.0, None, 0, None) == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_frame_composite_workspace_size(1, 20, 16, 880, 112) >= 20 * 16 * 80000
    assert gdn.gdn_frame_composite_workspace_size(1, 20, 0, 880, 112) == 0
    cmp_ = L.gdn_state_compose
    assert cmp_(None, None, fake, fake, 4, 112, None) == gdn.GDN_ERR_INVALID_ARG
    assert cmp_(None, fake, fake, fake, 4, 96, None) == gdn.GDN_ERR_UNSUPPORTED
    assert cmp_(None, fake, fake, fake, -1, 112, None) == gdn.GDN_ERR_INVALID_ARG
    assert cmp_(None, fake, fake, fake, 0, 112, None) == gdn.GDN_OK
    assert cmp_(P(0x10008), fake, fake, fake, 4, 112, None) == gdn.GDN_ERR_INVALID_ARG
    f32 = L.gdn_frame_fwd_f32
    assert f32(fake, fake, fake, fake, fake, None, fake, fake, 1, 1, 1, 1, 129, 0.0, None) == gdn.GDN_ERR_UNSUPPORTED
    assert f32(fake, fake, fake, fake, fake, None, fake, fake, 1, -1, 1, 1, 16, 0.0, None) == gdn.GDN_ERR_INVALID_ARG
    assert f32(None, fake, fake, fake, fake, None, fake, fake, 1, 1, 1, 1, 16, 0.0, None) == gdn.GDN_ERR_INVALID_ARG


def test_noalloc_step_statuses_match_frame_fwd(L):
    """The scratch-free step reports, for every argument list, the status gdn_frame_fwd
    (F = 1) reports when given a workspace of the scratch array's size, before any CUDA call:
    bad sizes, unsupported head sizes, null or misaligned pointers, shapes the size plan
    refuses, and requests larger than the array."""
    from gated_deltanet_wise_b300 import gdn
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every case below is refused on the host
    limit = L.gdn_frame_step_noalloc_limit_bytes()
    base = dict(q=fake, k=fake, v=fake, beta=fake, gamma=fake, S_in=None, S_out=fake, o=fake)
    cases = [
        ((-1, 1, 8, 112), {}), ((1, -2, 8, 112), {}), ((1, 1, -8, 112), {}), ((1, 1, 8, 0), {}),
        ((1, 1, 8, -112), {}), ((1, 1, 8, 64), {}), ((1, 1, 8, 128), {}), ((-1, 1, 8, 64), {}),
        ((1, 1, 8, 112), dict(q=None)), ((1, 1, 8, 112), dict(k=P(0x10008))),
        ((1, 1, 8, 112), dict(beta=P(0x10002))), ((1, 1, 8, 112), dict(S_in=P(0x10004))),
        ((1, (1 << 20) + 1, 8, 112), {}),                  # more chains than the size plan takes
        ((1, (1 << 20) + 1, 8, 112), dict(o=None)),        # ... with a bad pointer: the pointer first
        ((4, 40, 880, 112), {}),                           # 160 chains: larger than the array
        ((4, 40, 880, 112), dict(v=None)),
    ]
    for (B, H, N, D), over in cases:
        a = dict(base, **over)
        ptrs = (a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["S_in"], a["S_out"], a["o"])
        st_na = L.gdn_frame_step_noalloc(*ptrs, B, H, N, D, 0.0, None)
        st_fw = L.gdn_frame_fwd(*ptrs, B, H, 1, N, D, 0.0, fake, limit, None)
        assert st_na == st_fw, ((B, H, N, D), over, st_na, st_fw)
        assert st_na != gdn.GDN_OK, ((B, H, N, D), over)
    assert L.gdn_frame_step_noalloc(*(fake,) * 5, None, fake, fake, 4, 40, 880, 112, 0.0, None) == \
        gdn.GDN_ERR_WORKSPACE
    assert L.gdn_frame_step_noalloc(*(fake,) * 5, None, fake, fake, 1, (1 << 20) + 1, 8, 112, 0.0, None) == \
        gdn.GDN_ERR_UNSUPPORTED


def test_backward_frame_limit_refused_on_host(L):
    """Runs of 65,535 frames or more exceed a grid dimension of the backward's per-frame
    kernels: refused before anything is enqueued, and the size query says so."""
    from gated_deltanet_wise_b300 import gdn
    P = ctypes.c_void_p
    fake = P(0x10000)
    assert gdn.gdn_frame_bwd_workspace_size(1, 1, 65535, 8, 112) == 2 ** 64 - 1
    assert gdn.gdn_frame_bwd_workspace_size(1, 1, 65534, 8, 112) not in (0, 2 ** 64 - 1)
    st = L.gdn_frame_bwd(fake, fake, fake, fake, fake, None, fake, None, fake, fake, fake, fake, fake, None,
                         1, 1, 65535, 8, 112, 0.0, fake, 1 << 40, None)
    assert st == gdn.GDN_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from gated_deltanet_wise_b300 import gdn
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        gdn.lib()


def test_plain_c_consumer(L, tmp_path):
    """include/gdn.h compiles as C (gcc, no CUDA headers) and a C program linked
    against the library runs its host-side entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    from gated_deltanet_wise_b300 import build
    libdir = os.path.dirname(build.LIB)
    exe = str(tmp_path / "abi_consumer")
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-o", exe, "-L", libdir,
                           "-l:" + os.path.basename(build.LIB), "-Wl,-rpath," + libdir])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi consumer ok" in r.stdout
