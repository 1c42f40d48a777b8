"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest
import torch

from selective_state_space_138_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ss_scan.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(binding.EXPORTS)


def declared_arity():
    """Number of parameters of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(ss_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argtypes_match_the_header(lib):
    """Every function the binding declares argument types for takes as many
    arguments as the header says (a miscount would pass the wrong values)."""
    arity = declared_arity()
    assert set(arity) == set(binding.EXPORTS)
    for name, n in arity.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None, name
        assert len(argtypes) == n, (name, len(argtypes), n)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen("nm -D --defined-only %s" % binding.LIB_PATH).read()
    for name in declared_functions():
        assert re.search(r"\bT %s$" % name, out, flags=re.M), name


def test_abi_version_and_empty_error(lib):
    assert binding.abi_version() == 2
    assert isinstance(binding.last_error(), str)


def test_library_has_no_torch_dependency(lib):
    out = os.popen("ldd %s" % binding.LIB_PATH).read()
    assert "torch" not in out and "c10" not in out


@pytest.mark.gpu
def test_library_kernels_are_sm103a_binaries(lib):
    """The CUDA runtime loads the library's kernels as sm_103 binaries (the
    module's own record, read through an exported query), not a JIT of PTX."""
    assert binding.kernel_binary_version() == 103


def test_binary_version_query_needs_an_output(lib):
    assert lib.ss_kernel_binary_version(None) == -1


NULL = None


def _scan(lib, sfx, x=1, dt=1, A=1, B=1, C=1, y=1, batch=1, d=1, L=1, N=16):
    p = lambda v: ctypes.c_void_p(v) if v else None
    fn = getattr(lib, "ss_scan_fwd_" + sfx)
    return fn(p(x), p(dt), p(A), p(B), p(C), None, None, None, 1, p(y), None, batch, d, L, N, None)


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_scan_host_validation(lib, sfx):
    assert _scan(lib, sfx, batch=0) == -2
    assert _scan(lib, sfx, L=-3) == -2
    assert "positive" in binding.last_error()
    assert _scan(lib, sfx, N=0) == -3
    assert _scan(lib, sfx, N=65) == -3
    assert "N=65" in binding.last_error()
    assert _scan(lib, sfx, x=0) == -1
    assert "x" in binding.last_error()
    assert _scan(lib, sfx, y=0) == -1
    assert _scan(lib, sfx, batch=1 << 30, d=1 << 30, L=1 << 20) == -2


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_update_host_validation(lib, sfx):
    fn = getattr(lib, "ss_state_update_" + sfx)
    one = ctypes.c_void_p(1)
    assert fn(one, one, one, one, one, one, None, None, one, 0, 4, 16, None) == -2
    assert fn(one, one, one, one, one, one, None, None, one, 2, 4, 100, None) == -3
    assert fn(None, one, one, one, one, one, None, None, one, 2, 4, 16, None) == -1
    assert "state" in binding.last_error()


def test_binding_checks_shapes_before_calling():
    x = torch.zeros(2, 3, 8)
    with pytest.raises(ValueError):
        binding.scan_fwd(x, torch.zeros(2, 3, 9), torch.zeros(3, 4), torch.zeros(2, 4, 8), torch.zeros(2, 4, 8))
    with pytest.raises(TypeError):
        binding.scan_fwd(x.half(), x.half(), torch.zeros(3, 4), torch.zeros(2, 4, 8).half(),
                         torch.zeros(2, 4, 8).half())
    with pytest.raises(TypeError):
        binding.scan_fwd(x, x, torch.zeros(3, 4, dtype=torch.float64), torch.zeros(2, 4, 8),
                         torch.zeros(2, 4, 8))


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_conv_host_validation(lib, sfx):
    one = ctypes.c_void_p(1)
    fn = getattr(lib, "ss_causal_conv1d_" + sfx)
    assert fn(one, one, None, None, 1, one, None, 1, 4, 16, 9, None) == -2
    assert "k=9" in binding.last_error()
    assert fn(one, one, None, None, 1, one, None, 1, 4, 16, 0, None) == -2
    assert fn(None, one, None, None, 1, one, None, 1, 4, 16, 4, None) == -1
    assert fn(one, one, None, None, 1, one, None, 0, 4, 16, 4, None) == -2
    step = getattr(lib, "ss_conv_state_update_" + sfx)
    assert step(None, one, one, None, 1, one, 2, 4, 4, None) == -1
    assert "conv_state" in binding.last_error()
    assert step(one, one, one, None, 1, one, 2, 4, 12, None) == -2


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_bwd_host_validation(lib, sfx):
    one = ctypes.c_void_p(1)
    fn = getattr(lib, "ss_scan_bwd_" + sfx)

    def call(x=one, ws=one, ws_bytes=1 << 40, batch=2, d=4, L=16, N=16, dout=one):
        return fn(x, one, one, one, one, None, None, None, 1, None, dout, None, one, one, one, one, one,
                  None, None, None, None, ws, ws_bytes, 0, batch, d, L, N, None)

    assert call(batch=0) == -2
    assert call(N=33) == -3
    assert "N=33" in binding.last_error()
    assert call(x=None) == -1
    assert call(dout=None) == -1
    assert "dout" in binding.last_error()
    assert call(ws=None) == -1
    assert "workspace" in binding.last_error()


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_bwd_ex_host_validation(lib, sfx):
    """The backward of the scan variants checks its arguments like the plain
    one, before anything reaches a GPU."""
    one = ctypes.c_void_p(1)
    fn = getattr(lib, "ss_scan_bwd_ex_" + sfx)

    def call(x=one, ws=one, ws_bytes=1 << 40, batch=2, d=4, L=16, N=16, dout=one, starts=None, reverse=1):
        return fn(x, one, one, one, one, None, None, None, 1, None, starts, reverse, dout, None, one, one, one,
                  one, one, None, None, None, None, ws, ws_bytes, batch, d, L, N, None)

    assert call(batch=0) == -2
    assert call(N=33, starts=one) == -3
    assert call(x=None) == -1
    assert call(dout=None, reverse=0, starts=one) == -1
    assert "dout" in binding.last_error()
    assert call(ws=None) == -1


def test_device_faults_needs_an_output(lib):
    assert lib.ss_device_faults(None, 0) == -1
    assert "flags" in binding.last_error()


def test_bwd_workspace_size(lib):
    ws = binding.scan_bwd_workspace_bytes
    # one 16-byte state group (4 states) per channel and batch row at every 16th step
    assert ws(8, 1536, 2048, 16) == 8 * 1536 * (2048 // 16) * 4 * 16
    assert ws(1, 1, 17, 1) == 2 * 16
    assert ws(2, 3, 16, 20) == 2 * 3 * 1 * 8 * 16
    assert ws(1, 1, 1, 33) == 0 and ws(0, 1, 1, 1) == 0


def test_ssd_workspace_size(lib):
    ws = binding.ssd_workspace_bytes
    up = lambda v: (v + 255) // 256 * 256

    def expect(batch, L, H, G, N):
        chunks = (L + 63) // 64
        # C B^T of every chunk (bf16 64 x 64 per batch row, chunk and group), the chunk
        # walk's counters (one claim counter, one flag per row), the states handed
        # between a row's chunk segments (fp32 headdim 64 x N per row)
        return up(batch * chunks * G * 64 * 64 * 2) + up((1 + batch * H) * 4) + batch * H * 64 * N * 4

    assert ws(8, 2048, 80, 1, 128) == expect(8, 2048, 80, 1, 128)
    assert ws(1, 1, 1, 1, 64) == expect(1, 1, 1, 1, 64)
    assert ws(2, 130, 8, 4, 256) == expect(2, 130, 8, 4, 256)
    assert ws(0, 1, 1, 1, 64) == 0 and ws(1, 1, 1, 2, 64) == 0 and ws(1, 1, 1, 1, 512) == 0
    assert ws(1 << 40, 1 << 40, 1, 1, 64) == 0


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_bwd_noalloc_host_validation(lib, sfx):
    one = ctypes.c_void_p(1)
    fn = getattr(lib, "ss_scan_bwd_noalloc_" + sfx)

    def call(x=one, batch=2, d=4, L=16, N=16):
        return fn(x, one, one, one, one, None, None, None, 1, None, one, None, one, one, one, one, one,
                  None, None, None, None, batch, d, L, N, None)

    assert call(x=None) == -1
    assert call(N=33) == -3
    assert call(batch=0) == -2
    # the headline layer's stored states (about 100 MB) exceed the built-in scratch
    assert call(batch=8, d=1536, L=2048, N=16) == -2
    assert "built-in scratch" in binding.last_error()
    assert binding.scan_bwd_workspace_bytes(8, 1536, 2048, 16) > binding.BWD_NOALLOC_MAX_BYTES
    # sizes whose element count overflows are rejected before any size product is formed
    big = 1 << 40
    assert call(batch=big, d=big, L=big, N=16) == -2
    assert "overflows" in binding.last_error()
    assert binding.scan_bwd_workspace_bytes(big, big, big, 16) == 0
    assert binding.scan_bwd_workspace_bytes(1 << 20, 1 << 20, 1 << 20, 32) == 0


@pytest.mark.parametrize("sfx", ["bf16", "f32"])
def test_fwd_train_host_validation(lib, sfx):
    one = ctypes.c_void_p(1)
    fn = getattr(lib, "ss_scan_fwd_train_" + sfx)

    def call(ws=one, ws_bytes=1 << 40, N=16):
        return fn(one, one, one, one, one, None, None, None, 1, None, one, None, ws, ws_bytes, 2, 4, 16, N, None)

    assert call(ws=None) == -1
    assert "workspace" in binding.last_error()
    assert call(N=40) == -3
