"""The C-ABI library on the host: it loads, exports every entry point the
header declares, and its host-side logic (capacities, workspace sizing,
argument and state checks, options) behaves as specified. Nothing here runs a
kernel or needs a GPU."""
import ctypes as C
import os
import re

import pytest

from combine_ep_route_gb300 import _lib as L
from oracle import ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")
FAKE_WS = 0x7F0000000000   # a 256-aligned address; never dereferenced by these tests


@pytest.fixture(scope="module")
def lib():
    from combine_ep_route_gb300 import build
    build.build()
    return L.lib()


def cfg(W=8, E=64, K=8, T=128, h=2048, extras=(), flags=0, n_extra=None, x_dtype=None):
    c = L.EpConfigC()
    c.W, c.E, c.top_k, c.max_tokens, c.hidden = W, E, K, T, h
    c.x_dtype = L.EP_BF16 if x_dtype is None else x_dtype
    c.n_extra = len(extras) if n_extra is None else n_extra
    for i, b in enumerate(extras):
        c.extra_row_bytes[i] = b
    c.flags = flags
    return c


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|const char \*)\s*(ep_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, n


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name, val in re.findall(r"^#define (EP_\w+) (-?\d+)u?\b", text, re.M):
        if hasattr(L, name):
            assert getattr(L, name) == int(val), name


@pytest.mark.parametrize("W,E,K,T", [(2, 8, 2, 16), (8, 64, 8, 128), (4, 8, 8, 16), (32, 256, 8, 256),
                                     (1, 4, 2, 5), (64, 1024, 16, 3)])
def test_capacities_match_oracle(lib, W, E, K, T):
    a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
    assert lib.ep_capacities(C.byref(cfg(W, E, K, T, 128)), C.byref(a), C.byref(b), C.byref(c)) == 0
    assert (a.value, b.value, c.value) == ref.capacities(W, E, K, T)


@pytest.mark.parametrize("bad", [
    dict(W=0), dict(W=65, E=1040), dict(E=60), dict(E=2048), dict(K=0), dict(K=17), dict(T=0),
    dict(h=4), dict(h=12), dict(extras=(20,)), dict(extras=(16,) * 4, n_extra=5), dict(n_extra=-1), dict(flags=8),
    dict(h=60000), dict(W=64, E=1024, T=40000), dict(K=2, flags=4),
    dict(x_dtype=9), dict(x_dtype=L.EP_FP8, h=24), dict(x_dtype=L.EP_FP4X2, h=40),
    dict(K=1, flags=4, x_dtype=L.EP_FP8),
])
def test_invalid_configs_rejected(lib, bad):
    n = C.c_size_t()
    c = cfg(**bad)
    assert lib.ep_workspace_bytes(C.byref(c), C.byref(n)) == L.EP_ERR_INVALID_ARG
    a = C.c_int32()
    assert lib.ep_capacities(C.byref(c), C.byref(a), C.byref(a), C.byref(a)) == L.EP_ERR_INVALID_ARG
    h = C.c_void_p()
    assert lib.ep_ctx_create(C.byref(c), C.c_void_p(FAKE_WS), 1 << 40, C.byref(h)) == L.EP_ERR_INVALID_ARG


def test_quantised_row_types_size_the_send_rows(lib):
    for xd, rb in [(L.EP_BF16, 4096), (L.EP_FP8, 2048), (L.EP_FP4X2, 1024)]:
        h, _ = _ctx(lib, cfg(x_dtype=xd, extras=(128,), flags=L.EP_FLAG_SENDBUF))
        m = L.EpMetadataC()
        assert lib.ep_get_metadata(h, C.byref(m)) == 0
        assert m.row_bytes == rb + 128
        lib.ep_ctx_destroy(h)


def test_workspace_sizing(lib):
    n1, n2 = C.c_size_t(), C.c_size_t()
    assert lib.ep_workspace_bytes(C.byref(cfg()), C.byref(n1)) == 0
    assert lib.ep_workspace_bytes(C.byref(cfg(flags=L.EP_FLAG_SENDBUF)), C.byref(n2)) == 0
    assert n1.value % 256 == 0
    # the send-buffer path adds the send and receive rank blocks
    assert n2.value - n1.value >= 2 * 8 * 8 * 128 * 4096
    n3 = C.c_size_t()
    assert lib.ep_workspace_bytes(C.byref(cfg(extras=(128,), flags=L.EP_FLAG_SENDBUF)), C.byref(n3)) == 0
    assert n3.value - n2.value >= 2 * 8 * 8 * 128 * 128


def _ctx(lib, c=None):
    c = c or cfg()
    n = C.c_size_t()
    assert lib.ep_workspace_bytes(C.byref(c), C.byref(n)) == 0
    h = C.c_void_p()
    assert lib.ep_ctx_create(C.byref(c), C.c_void_p(FAKE_WS), n.value, C.byref(h)) == 0
    return h, n.value


def test_ctx_create_checks_workspace(lib):
    c = cfg()
    n = C.c_size_t()
    lib.ep_workspace_bytes(C.byref(c), C.byref(n))
    h = C.c_void_p()
    assert lib.ep_ctx_create(C.byref(c), None, n.value, C.byref(h)) == L.EP_ERR_INVALID_ARG
    assert lib.ep_ctx_create(C.byref(c), C.c_void_p(FAKE_WS + 16), n.value, C.byref(h)) == L.EP_ERR_WORKSPACE
    assert lib.ep_ctx_create(C.byref(c), C.c_void_p(FAKE_WS), n.value - 1, C.byref(h)) == L.EP_ERR_WORKSPACE
    assert lib.ep_ctx_destroy(None) == 0


def test_host_side_argument_and_state_checks(lib):
    h, nbytes = _ctx(lib)
    p = C.c_void_p(FAKE_WS)
    # combine before any dispatch: refused before any GPU work
    assert lib.ep_combine(h, p, L.EP_BF16, p, None) == L.EP_ERR_STATE
    assert lib.ep_combine(h, p, 7, p, None) == L.EP_ERR_INVALID_ARG
    assert lib.ep_combine(h, None, L.EP_BF16, p, None) == L.EP_ERR_INVALID_ARG
    assert lib.ep_combine(h, C.c_void_p(FAKE_WS + 8), L.EP_BF16, p, None) == L.EP_ERR_INVALID_ARG
    # dispatch argument checks happen before any GPU work
    args = [h, p, None, p, p, None, p, None, p]
    assert lib.ep_dispatch(*args, 5, None) == L.EP_ERR_INVALID_ARG
    assert lib.ep_dispatch(*args, L.EP_PATH_SENDBUF, None) == L.EP_ERR_WORKSPACE
    bad = list(args)
    bad[1] = C.c_void_p(FAKE_WS + 2)
    assert lib.ep_dispatch(*bad, L.EP_PATH_FUSED, None) == L.EP_ERR_INVALID_ARG
    bad = list(args)
    bad[3] = None
    assert lib.ep_dispatch(*bad, L.EP_PATH_FUSED, None) == L.EP_ERR_INVALID_ARG
    # status before any dispatch touches nothing
    assert lib.ep_status(h, None) == 0
    assert lib.ep_ctx_reset(h) == 0
    assert lib.ep_ctx_destroy(h) == 0


def test_two_stage_combine_host_checks(lib):
    p = C.c_void_p(FAKE_WS)
    h, _ = _ctx(lib)                                  # no send-buffer workspace
    assert lib.ep_combine_two_stage(h, p, L.EP_BF16, p, None) == L.EP_ERR_WORKSPACE
    lib.ep_ctx_destroy(h)
    h, _ = _ctx(lib, cfg(flags=L.EP_FLAG_SENDBUF))
    assert lib.ep_combine_two_stage(h, p, L.EP_BF16, p, None) == L.EP_ERR_STATE
    assert lib.ep_combine_two_stage(h, p, 3, p, None) == L.EP_ERR_INVALID_ARG
    lib.ep_ctx_destroy(h)


def test_extra_payload_pointers_required(lib):
    h, _ = _ctx(lib, cfg(extras=(128,)))
    p = C.c_void_p(FAKE_WS)
    assert lib.ep_dispatch(h, p, None, p, p, None, p, None, p, L.EP_PATH_FUSED, None) == L.EP_ERR_INVALID_ARG
    arr = (C.c_void_p * 1)(None)
    assert lib.ep_dispatch(h, p, None, p, p, arr, p, arr, p, L.EP_PATH_FUSED, None) == L.EP_ERR_INVALID_ARG
    lib.ep_ctx_destroy(h)


def test_options(lib):
    h, _ = _ctx(lib)
    ok = [(L.EP_OPT_WAIT_LIMIT_NS, 10**6), (L.EP_OPT_KERNEL_TIMING, 1), (L.EP_OPT_PDL, 0),
          (L.EP_OPT_MOVE_CTAS_PER_SM, 2), (L.EP_OPT_MOVE_PIPES, 8), (L.EP_OPT_FAULT_SKIP_PUBLISH, 0),
          (L.EP_OPT_FAULT_SKIP_PUBLISH, -1), (L.EP_OPT_COMBINE_CTAS_PER_SM, 4),
          (L.EP_OPT_COMBINE_CTAS_PER_SM, 0), (L.EP_OPT_MOVE_CHUNK_BYTES, 4096),
          (L.EP_OPT_MOVE_CHUNK_BYTES, 0), (L.EP_OPT_MOVE_MAX_STAGES, 16), (L.EP_OPT_FUSED_DISPATCH, 0),
          (L.EP_OPT_FUSED_DISPATCH, 1), (L.EP_OPT_ROUTE_CTAS, 0), (L.EP_OPT_ROUTE_CTAS, 16),
          (L.EP_OPT_MOVE_PIPES, -1), (L.EP_OPT_MOVE_CHUNK_BYTES, -1), (L.EP_OPT_MOVE_MAX_STAGES, -1),
          (L.EP_OPT_ROUTE_CTAS, -1)]
    for o, v in ok:
        assert lib.ep_set_option(h, o, v) == 0, (o, v)
    bad = [(0, 1), (99, 1), (L.EP_OPT_WAIT_LIMIT_NS, 10), (L.EP_OPT_KERNEL_TIMING, 2),
           (L.EP_OPT_MOVE_CTAS_PER_SM, 0), (L.EP_OPT_MOVE_PIPES, 9), (L.EP_OPT_FAULT_SKIP_PUBLISH, 10**6),
           (L.EP_OPT_MOVE_CHUNK_BYTES, 100), (L.EP_OPT_MOVE_MAX_STAGES, 1), (L.EP_OPT_COMBINE_CTAS_PER_SM, 17),
           (L.EP_OPT_ROUTE_CTAS, -2), (L.EP_OPT_ROUTE_CTAS, 4097), (L.EP_OPT_MOVE_PIPES, -2),
           (L.EP_OPT_MOVE_PIPES, 0), (L.EP_OPT_MOVE_CHUNK_BYTES, -16), (L.EP_OPT_MOVE_MAX_STAGES, -2)]
    for o, v in bad:
        assert lib.ep_set_option(h, o, v) == L.EP_ERR_INVALID_ARG, (o, v)
    kt = L.EpKernelTimesC()
    assert lib.ep_kernel_times(h, C.byref(kt)) == 0
    assert all(kt.launches[i] == 0 for i in range(L.EP_K_COUNT))
    lib.ep_ctx_destroy(h)


def test_metadata_lives_inside_the_workspace(lib):
    c = cfg(extras=(64,), flags=L.EP_FLAG_SENDBUF)
    h, nbytes = _ctx(lib, c)
    m = L.EpMetadataC()
    assert lib.ep_get_metadata(h, C.byref(m)) == 0
    ptrs = [m.send_cnt, m.pair_row, m.pair_w, m.pair_send, m.recv_eloc, m.recv_w, m.recv_row,
            m.send_x, m.recv_x]
    assert len(set(ptrs)) == len(ptrs)
    for q in ptrs:
        assert FAKE_WS <= q < FAKE_WS + nbytes and q % 256 == 0
    assert m.slots_per_token == 8 and m.expert_cap == 1024 and m.row_bytes == 4096 + 64
    lib.ep_ctx_destroy(h)


def test_error_strings(lib):
    for code in range(0, -9, -1):
        s = lib.ep_error_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ep_error_string(-100).decode() == "unknown status"


def test_agrs_host_checks(lib):
    """ep_agrs refuses what it cannot run before touching any GPU."""
    p = C.c_void_p(FAKE_WS)
    b = L.EpAgrsBuffersC(FAKE_WS, FAKE_WS, FAKE_WS, FAKE_WS, None)

    def call(c=None, a1=p, ids=p, w=p, buf=b, dt=L.EP_BF16, out=p):
        return lib.ep_agrs(C.byref(c if c is not None else cfg(W=4, E=16, K=4, T=64, h=512)), None,
                           a1, ids, w, C.byref(buf) if buf is not None else None, dt, out, None)

    assert call(c=cfg(W=3, E=16)) == L.EP_ERR_INVALID_ARG                 # E % W != 0
    assert call(c=cfg(W=4, E=16, K=4, T=64, h=512, x_dtype=L.EP_FP8)) == L.EP_ERR_INVALID_ARG
    assert call(c=cfg(W=4, E=16, K=1, T=64, h=512,
                      flags=L.EP_FLAG_WEIGHT_ON_INPUT)) == L.EP_ERR_INVALID_ARG
    assert call(dt=3) == L.EP_ERR_INVALID_ARG
    assert call(a1=None) == L.EP_ERR_INVALID_ARG
    assert call(out=None) == L.EP_ERR_INVALID_ARG
    assert call(buf=None) == L.EP_ERR_INVALID_ARG
    assert call(buf=L.EpAgrsBuffersC(FAKE_WS, None, FAKE_WS, FAKE_WS, None)) == L.EP_ERR_INVALID_ARG
    assert call(a1=C.c_void_p(FAKE_WS + 8)) == L.EP_ERR_INVALID_ARG      # rows need 16-byte alignment
    assert call(buf=L.EpAgrsBuffersC(FAKE_WS, FAKE_WS, FAKE_WS, FAKE_WS + 4, None)) == L.EP_ERR_INVALID_ARG
    # W^2 * Tm * h / 8 work items must stay below 2^31
    assert call(c=cfg(W=64, E=64, K=8, T=8192, h=512)) == L.EP_ERR_INVALID_ARG


@pytest.mark.parametrize("lang,std", [("c", "c89"), ("c", "c99"), ("c", "c11"), ("c++", "c++17")])
def test_header_compiles_alone_with_strict_warnings(tmp_path, lang, std):
    """include/ep.h is plain C: it needs no CUDA or torch header and compiles
    without a warning as C89 through C11 and as C++."""
    import shutil
    import subprocess
    cc = "gcc" if lang == "c" else "g++"
    if shutil.which(cc) is None:
        pytest.skip(f"{cc} not available")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "ep.h"\nint main(void) { return EP_OK; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_launches_only_on_the_buffers_device(monkeypatch):
    """The binding refuses to enqueue when the current CUDA device (where the
    library launches) is not the device the buffers live on, or when the given
    stream belongs to another device: such a launch would address another
    device's memory. Checked with a fake current device, no GPU needed."""
    import torch
    from combine_ep_route_gb300 import ep

    class FakeStream:
        def __init__(self, idx):
            self.device = torch.device("cuda", idx)
            self.cuda_stream = 1234 + idx

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: FakeStream(0))
    assert ep._stream_ptr(None, torch.device("cuda", 0)) == 1234
    assert ep._stream_ptr(FakeStream(0), torch.device("cuda", 0)) == 1234
    with pytest.raises(ValueError, match="current device"):
        ep._stream_ptr(None, torch.device("cuda", 1))
    with pytest.raises(ValueError, match="current device"):
        ep._stream_ptr(None, torch.device("cpu"))          # host buffers never reach a kernel
    with pytest.raises(ValueError, match="stream is on"):
        ep._stream_ptr(FakeStream(1), torch.device("cuda", 0))
    assert ep._cuda_device(None) == torch.device("cuda", 0)
    assert ep._cuda_device("cuda") == torch.device("cuda", 0)
    assert ep._cuda_device(torch.device("cuda", 3)) == torch.device("cuda", 3)
    with pytest.raises(ValueError):
        ep._cuda_device("cpu")
