"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects invalid arguments before anything reaches a GPU.

Only argument combinations that fail host validation are passed here (fake,
never-dereferenced device addresses); no call in this file launches work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = []
    for fname in sorted(os.listdir(HEADER_DIR)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(sp_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_entry_points():
    names = _declared_functions()
    for must in ("sp_rs_norm_fwd", "sp_allgather_seq", "sp_norm_bwd",
                 "sp_norm_bwd_workspace_bytes", "sp_reduce_scatter_seq"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.sp_abi_version() == 1


FAKE = 0x7F0000000000          # 16-byte aligned, never dereferenced


def _arr(vals):
    a = (ctypes.c_void_p * max(1, len(vals)))(*vals)
    return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))


def _fwd_args(**kw):
    t = kw.get("t", 2)
    b, s, h = kw.get("b", 1), kw.get("s", 8), kw.get("h", 64)
    n_gather = kw.get("n_gather", 1)
    step = 1 << 24
    base = FAKE
    nxt = iter(range(base, base + 200 * step, step))
    part = kw.get("partials", [next(nxt) for _ in range(t)])
    res = [next(nxt) for _ in range(t)]
    z = kw.get("z", [next(nxt) for _ in range(t)])
    mask = [next(nxt) for _ in range(t)]
    mean = [next(nxt) for _ in range(t)]
    rstd = [next(nxt) for _ in range(t)]
    gath = kw.get("gathered", [next(nxt) for _ in range(n_gather)])
    bias, gamma, beta = next(nxt), next(nxt), next(nxt)
    return [_arr(part), _arr(res), ctypes.c_void_p(bias), ctypes.c_void_p(gamma),
            ctypes.c_void_p(beta), b, s, h, t, kw.get("eps", 1e-5), kw.get("p", 0.1), 1234, 0,
            kw.get("cu", None), kw.get("n_seqs", 0), kw.get("norm", 0), _arr(z), _arr(mask),
            _arr(mean), _arr(rstd), _arr(gath), n_gather, None, None]


@pytest.mark.parametrize("kw,code", [
    (dict(t=0), 1), (dict(t=17), 1), (dict(h=12), 1), (dict(h=0), 1), (dict(s=9), 1),
    (dict(h=16392), 3), (dict(p=1.0), 1), (dict(p=-0.5), 1), (dict(eps=0.0), 1),
    (dict(eps=float("nan")), 1), (dict(n_gather=17), 1), (dict(norm=5), 1),
    (dict(partials=[FAKE + 8, FAKE + (1 << 30)]), 2),
    (dict(partials=[0, FAKE + (1 << 30)]), 1),
    (dict(b=2, cu=ctypes.c_void_p(FAKE), n_seqs=2), 1),
    (dict(cu=ctypes.c_void_p(FAKE), n_seqs=0), 1),
    # the gathered output placed on top of rank 0's partial
    (dict(gathered=[FAKE]), 7),
    # two shards' Z outputs at the same address
    (dict(z=[FAKE + (3 << 30), FAKE + (3 << 30)]), 7),
])
def test_forward_rejects_invalid_arguments(lib, kw, code):
    lib.sp_rs_norm_fwd.restype = ctypes.c_int32
    lib.sp_rs_norm_fwd.argtypes = [
        ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int32, ctypes.c_float, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64,
        ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32] + [ctypes.POINTER(ctypes.c_void_p)] * 5 + [
        ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    got = lib.sp_rs_norm_fwd(*_fwd_args(**kw))
    assert got == code, lib.sp_last_error()
    lib.sp_last_error.restype = ctypes.c_char_p
    assert lib.sp_last_error()


def test_backward_and_collectives_reject_invalid_arguments():
    from sp_boundary_norm_gb300 import binding
    lib = binding.load()
    arr = _arr([FAKE, FAKE + (1 << 30)])
    # t out of range
    assert lib.sp_allgather_seq(arr, 1, 8, 64, 0, None, 0, arr, 1, None, None) == 1
    # n_gather 0 is not a gather
    assert lib.sp_allgather_seq(arr, 1, 8, 64, 2, None, 0, arr, 0, None, None) == 1
    # misaligned shard
    bad = _arr([FAKE + 4, FAKE + (1 << 30)])
    assert lib.sp_reduce_scatter_seq(bad, 1, 8, 64, 2, None, 0, arr, None, None) == 2
    # backward: p out of range, then a missing workspace
    six = [arr] * 5
    r = lib.sp_norm_bwd(arr, arr, arr, arr, arr, ctypes.c_void_p(FAKE), None, 1, 8, 64, 2, 1.5,
                        None, 0, 0, arr, arr, 1, None, None, None, None, 0, None, None)
    assert r == 1
    out = _arr([FAKE + (5 << 30), FAKE + (6 << 30)])
    r = lib.sp_norm_bwd(_arr([FAKE, FAKE + (1 << 28)]), _arr([FAKE + (1 << 29), FAKE + (3 << 28)]),
                        _arr([FAKE + (1 << 31), FAKE + (5 << 28)]),
                        _arr([FAKE + (6 << 28), FAKE + (7 << 28)]),
                        _arr([FAKE + (9 << 28), FAKE + (10 << 28)]), ctypes.c_void_p(FAKE + (11 << 28)),
                        None, 1, 8, 64, 2, 0.1, None, 0, 0, out, _arr([FAKE + (8 << 30)]), 1,
                        None, None, None, None, 0, None, None)
    assert r == 1 and b"workspace" in lib.sp_last_error()
    del six


def test_injected_failure_is_returned_once(lib):
    from sp_boundary_norm_gb300 import binding
    lib = binding.load()
    assert lib.sp_debug_inject(5) == 0
    arr = _arr([FAKE, FAKE + (1 << 30)])
    assert lib.sp_allgather_seq(arr, 1, 8, 64, 0, None, 0, arr, 1, None, None) == 5
    assert b"injected" in lib.sp_last_error()
    # disarmed: the same call now fails validation instead
    assert lib.sp_allgather_seq(arr, 1, 8, 64, 0, None, 0, arr, 1, None, None) == 1


def test_last_shape_hook_host_rules(lib):
    """The shape hook is per thread: zeros before a thread's first call; bad
    kernel indices are rejected."""
    import threading
    from sp_boundary_norm_gb300 import binding
    binding.load()
    got = {}
    th = threading.Thread(target=lambda: got.update(binding.sp_debug_last_shape(0)))
    th.start()
    th.join()
    assert got == dict(threads=0, chunks=0, stages=0, grid=0, cluster=0, smem=0)
    with pytest.raises(binding.SpError):
        binding.sp_debug_last_shape(2)


def test_workspace_size_shape_rules(lib):
    from sp_boundary_norm_gb300 import binding
    binding.load()
    assert binding.sp_norm_bwd_workspace_bytes(1, 0, 64, 2) == 0
    n = binding.sp_norm_bwd_workspace_bytes(1, 64, 64, 2)
    assert n > 0 and n % (3 * 64 * 4) == 0
    assert binding.sp_norm_bwd_workspace_bytes(1, 64, 12, 2) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from sp_boundary_norm_gb300 import _build, binding
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.load()


def test_bit_mask_entry_points_validate_on_the_host():
    """The bit-packed mask needs h % 32 == 0 and a mask array; both are
    refused before anything is enqueued, by the forward and both backwards."""
    from sp_boundary_norm_gb300 import binding
    lib = binding.load()
    args = _fwd_args(h=520)
    assert lib.sp_rs_norm_fwd_bitmask(*args) == 3             # SP_ERR_UNSUPPORTED
    assert b"multiple of 32" in lib.sp_last_error()
    args = _fwd_args(h=512)
    args[17] = None                                           # the mask_bits_out array
    assert lib.sp_rs_norm_fwd_bitmask(*args) == 1             # SP_ERR_INVALID_ARG
    assert b"mask_bits_out" in lib.sp_last_error()
    arr = _arr([FAKE, FAKE + (1 << 30)])
    for fn in (lib.sp_norm_bwd_bitmask, lib.sp_rs_norm_bwd_bitmask):
        r = fn(arr, arr, arr, arr, arr, ctypes.c_void_p(FAKE), None, 1, 8, 520, 2, 0.1, None, 0,
               0, arr, arr, 1, None, None, None, None, 0, None, None)
        assert r == 3 and b"multiple of 32" in lib.sp_last_error()
    # the byte-mask forward accepts a NULL mask array (nothing stored): it
    # gets past the mask check and stops at the next invalid argument
    args = _fwd_args(h=512, p=1.5)
    args[17] = None
    assert lib.sp_rs_norm_fwd(*args) == 1 and b"p = " in lib.sp_last_error()
