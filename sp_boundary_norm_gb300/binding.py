"""Thin Python binding of ``libspboundary.so`` (ctypes; marshalling only).

The functions carry the C entry points' names.  They take torch tensors for
device memory, check shapes, dtypes and devices (the C ABI trusts the sizes
it is given), and pass raw pointers and the current CUDA stream.  Every step
of the boundary runs in the library's CUDA kernels; there is no fallback: if
the library is not built, ``load()`` raises.
"""
import contextlib
import ctypes
import os

import torch

from . import _build

SP_OK = 0
STATUS_NAMES = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_MISALIGNED",
                3: "SP_ERR_UNSUPPORTED", 4: "SP_ERR_CUDA", 5: "SP_ERR_TIMEOUT",
                6: "SP_ERR_DEVICE_CHECK", 7: "SP_ERR_OVERLAP"}
NORMS = {"layernorm": 0, "rmsnorm": 1}
MAX_RANKS = 16

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64
_PP = ctypes.POINTER(ctypes.c_void_p)

_lib = None


class SpError(RuntimeError):
    def __init__(self, code, message):
        self.code = code
        self.name = STATUS_NAMES.get(code, str(code))
        super().__init__(f"{self.name}: {message}")


def load():
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.sp_rs_norm_fwd.restype = _i32
    lib.sp_rs_norm_fwd.argtypes = [
        _PP, _PP, _vp, _vp, _vp, _i64, _i64, _i64, _i32, ctypes.c_float, ctypes.c_double,
        _u64, _u64, _vp, _i32, _i32, _PP, _PP, _PP, _PP, _PP, _i32, _vp, _vp]
    lib.sp_allgather_seq.restype = _i32
    lib.sp_allgather_seq.argtypes = [_PP, _i64, _i64, _i64, _i32, _vp, _i32, _PP, _i32, _vp, _vp]
    lib.sp_reduce_scatter_seq.restype = _i32
    lib.sp_reduce_scatter_seq.argtypes = [_PP, _i64, _i64, _i64, _i32, _vp, _i32, _PP, _vp, _vp]
    lib.sp_norm_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.sp_norm_bwd_workspace_bytes.argtypes = [_i64, _i64, _i64, _i32, _i32]
    lib.sp_norm_bwd.restype = _i32
    lib.sp_norm_bwd.argtypes = [
        _PP, _PP, _PP, _PP, _PP, _vp, _PP, _i64, _i64, _i64, _i32, ctypes.c_double, _vp, _i32,
        _i32, _PP, _PP, _i32, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
    lib.sp_shard_norm_fwd.restype = _i32
    lib.sp_shard_norm_fwd.argtypes = [
        _PP, _PP, _vp, _vp, _vp, _i64, _i64, _i64, _i32, ctypes.c_float, ctypes.c_double,
        _u64, _u64, _vp, _i32, _i32, _PP, _PP, _PP, _PP, _PP, _vp, _vp]
    lib.sp_rs_norm_bwd.restype = _i32
    lib.sp_rs_norm_bwd.argtypes = list(lib.sp_norm_bwd.argtypes)
    lib.sp_rs_norm_bwd_bitmask.restype = _i32
    lib.sp_rs_norm_bwd_bitmask.argtypes = list(lib.sp_norm_bwd.argtypes)
    lib.sp_norm_bwd_bitmask.restype = _i32
    lib.sp_norm_bwd_bitmask.argtypes = list(lib.sp_norm_bwd.argtypes)
    lib.sp_rs_norm_fwd_bitmask.restype = _i32
    lib.sp_rs_norm_fwd_bitmask.argtypes = list(lib.sp_rs_norm_fwd.argtypes)
    lib.sp_norm_bwd_philox.restype = _i32
    lib.sp_norm_bwd_philox.argtypes = [
        _PP, _PP, _PP, _PP, _vp, _PP, _i64, _i64, _i64, _i32, ctypes.c_double, _u64, _u64, _vp,
        _i32, _i32, _PP, _PP, _i32, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
    lib.sp_norm_bwd_noalloc.restype = _i32
    lib.sp_norm_bwd_noalloc.argtypes = [
        _PP, _PP, _PP, _PP, _PP, _vp, _PP, _i64, _i64, _i64, _i32, ctypes.c_double, _vp, _i32,
        _i32, _PP, _PP, _i32, _vp, _vp, _vp, _vp, _vp]
    lib.sp_last_error.restype = ctypes.c_char_p
    lib.sp_last_error.argtypes = []
    lib.sp_abi_version.restype = _i32
    lib.sp_abi_version.argtypes = []
    lib.sp_debug_inject.restype = _i32
    lib.sp_debug_inject.argtypes = [_i32]
    lib.sp_debug_tune.restype = _i32
    lib.sp_debug_tune.argtypes = [_i32, _i32, _i32, _i32, _i32]
    lib.sp_debug_last_shape.restype = _i32
    lib.sp_debug_last_shape.argtypes = [_i32, _vp]
    lib.sp_debug_philox.restype = _i32
    lib.sp_debug_philox.argtypes = [_vp, _vp, _i64, _vp]
    _lib = lib
    return lib


def _check(code):
    if code != SP_OK:
        msg = load().sp_last_error()
        raise SpError(code, msg.decode() if msg else "")


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _ptr_array(ts):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * max(1, len(ts)))()
    for i, x in enumerate(ts):
        arr[i] = x.data_ptr()
    return ctypes.cast(arr, _PP)


def _on_device(device):
    """The calls launch on the current CUDA device: make it the tensors' own."""
    return torch.cuda.device(device) if device.type == "cuda" else contextlib.nullcontext()


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(x, shape, dtype, device, what):
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if tuple(x.shape) != tuple(shape):
        raise ValueError(f"{what}: shape {tuple(x.shape)} != {tuple(shape)}")
    if x.dtype != dtype:
        raise ValueError(f"{what}: dtype {x.dtype} != {dtype}")
    if x.device != device:
        raise ValueError(f"{what}: on {x.device}, expected {device}")
    if not x.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")


def shard_sizes(s, t):
    """Tokens per shard along s: o_k = floor(k*s/t)."""
    o = [(k * s) // t for k in range(t + 1)]
    return [o[k + 1] - o[k] for k in range(t)]


_status = {}


def device_status(device):
    """The binding's device status word for ``device`` (an int32 tensor); a
    bare "cuda" means the current CUDA device, as it does for tensors."""
    device = torch.device(device)
    if device.type == "cuda" and device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    if device not in _status:
        _status[device] = torch.zeros(1, dtype=torch.int32, device=device)
    return _status[device]


def check_device_status(device, reset=True):
    """Raise SpError if a kernel flagged a device-side failure (synchronises)."""
    st = device_status(device)
    code = int(st.item())
    if reset:
        st.zero_()
    if code != SP_OK:
        raise SpError(code, "device-side check failed")


def _seq_meta(cu_seqlens, b, device):
    if cu_seqlens is None:
        return None, 0
    _need(cu_seqlens, (cu_seqlens.numel(),), torch.int32, device, "cu_seqlens")
    if b != 1:
        raise ValueError("cu_seqlens requires b == 1")
    return _ptr(cu_seqlens), cu_seqlens.numel() - 1


def sp_rs_norm_fwd(partials, residual, bias, gamma, beta, *, eps, p, seed, offset=0,
                   cu_seqlens=None, norm="layernorm", z_out, mask_out, mean_out, rstd_out,
                   gathered, status=None):
    """Fused g* + bias + dropout + residual + norm + g (writes the given outputs;
    mask_out=None stores no mask: the backward is then sp_norm_bwd_philox)."""
    _rs_norm_fwd_call("sp_rs_norm_fwd", 1, partials, residual, bias, gamma, beta, eps, p, seed,
                      offset, cu_seqlens, norm, z_out, mask_out, mean_out, rstd_out, gathered,
                      status)


def sp_rs_norm_fwd_bitmask(partials, residual, bias, gamma, beta, *, eps, p, seed, offset=0,
                           cu_seqlens=None, norm="layernorm", z_out, mask_bits_out, mean_out,
                           rstd_out, gathered, status=None):
    """sp_rs_norm_fwd storing the mask one bit per element
    (mask_bits_out[k]: (b, s_k, h / 8) uint8, bit e of byte j = channel 8j + e)."""
    if mask_bits_out is None:
        raise ValueError("mask_bits_out is required")
    _rs_norm_fwd_call("sp_rs_norm_fwd_bitmask", 8, partials, residual, bias, gamma, beta, eps,
                      p, seed, offset, cu_seqlens, norm, z_out, mask_bits_out, mean_out,
                      rstd_out, gathered, status)


def _rs_norm_fwd_call(entry, mask_div, partials, residual, bias, gamma, beta, eps, p, seed,
                      offset, cu_seqlens, norm, z_out, mask_out, mean_out, rstd_out, gathered,
                      status):
    lib = load()
    t = len(partials)
    if not 1 <= t <= MAX_RANKS:
        raise ValueError("1 <= t <= 16")
    b, s, h = partials[0].shape
    dev = partials[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    for r in range(t):
        _need(partials[r], (b, s, h), bf, dev, f"partials[{r}]")
    ln = norm == "layernorm"
    for k in range(t):
        _need(residual[k], (b, sizes[k], h), bf, dev, f"residual[{k}]")
        _need(z_out[k], (b, sizes[k], h), bf, dev, f"z_out[{k}]")
        if mask_out is not None:
            _need(mask_out[k], (b, sizes[k], h // mask_div), torch.uint8, dev, f"mask_out[{k}]")
        _need(rstd_out[k], (b, sizes[k]), torch.float32, dev, f"rstd_out[{k}]")
        if ln:
            _need(mean_out[k], (b, sizes[k]), torch.float32, dev, f"mean_out[{k}]")
    for j, g in enumerate(gathered):
        _need(g, (b, s, h), bf, dev, f"gathered[{j}]")
    for name, v in (("bias", bias), ("gamma", gamma)):
        _need(v, (h,), bf, dev, name)
    if ln:
        _need(beta, (h,), bf, dev, "beta")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        code = getattr(lib, entry)(
            _ptr_array(partials), _ptr_array(residual), _ptr(bias), _ptr(gamma),
            _ptr(beta) if ln else None, b, s, h, t, float(eps), float(p), int(seed), int(offset),
            cu, n_seqs, NORMS[norm], _ptr_array(z_out), _ptr_array(mask_out),
            _ptr_array(mean_out) if ln else None, _ptr_array(rstd_out), _ptr_array(gathered),
            len(gathered), _ptr(st), _stream(dev))
    _check(code)


def sp_shard_norm_fwd(y_shards, residual, bias, gamma, beta, *, s, eps, p, seed, offset=0,
                      cu_seqlens=None, norm="layernorm", z_out, mask_out, mean_out, rstd_out,
                      o_shards, status=None):
    """Unfused middle step: bias + dropout + residual + norm on reduced shards
    (mask_out=None: no mask stored, as for sp_rs_norm_fwd)."""
    lib = load()
    t = len(y_shards)
    b, _, h = y_shards[0].shape
    dev = y_shards[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    ln = norm == "layernorm"
    for k in range(t):
        for name, x in (("y_shards", y_shards), ("residual", residual), ("z_out", z_out),
                        ("o_shards", o_shards)):
            _need(x[k], (b, sizes[k], h), bf, dev, f"{name}[{k}]")
        if mask_out is not None:
            _need(mask_out[k], (b, sizes[k], h), torch.uint8, dev, f"mask_out[{k}]")
        _need(rstd_out[k], (b, sizes[k]), torch.float32, dev, f"rstd_out[{k}]")
        if ln:
            _need(mean_out[k], (b, sizes[k]), torch.float32, dev, f"mean_out[{k}]")
    for name, v in (("bias", bias), ("gamma", gamma)):
        _need(v, (h,), bf, dev, name)
    if ln:
        _need(beta, (h,), bf, dev, "beta")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        _check(lib.sp_shard_norm_fwd(
            _ptr_array(y_shards), _ptr_array(residual), _ptr(bias), _ptr(gamma),
            _ptr(beta) if ln else None, b, s, h, t, float(eps), float(p), int(seed), int(offset),
            cu, n_seqs, NORMS[norm], _ptr_array(z_out), _ptr_array(mask_out),
            _ptr_array(mean_out) if ln else None, _ptr_array(rstd_out), _ptr_array(o_shards),
            _ptr(st), _stream(dev)))


def sp_allgather_seq(shards, gathered, *, s, cu_seqlens=None, status=None):
    """g alone: gathered[j][:, o_k:o_{k+1}, :] = shards[k] for every j."""
    lib = load()
    t = len(shards)
    b, _, h = shards[0].shape
    dev = shards[0].device
    sizes = shard_sizes(s, t)
    for k in range(t):
        _need(shards[k], (b, sizes[k], h), torch.bfloat16, dev, f"shards[{k}]")
    for j, g in enumerate(gathered):
        _need(g, (b, s, h), torch.bfloat16, dev, f"gathered[{j}]")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        _check(lib.sp_allgather_seq(_ptr_array(shards), b, s, h, t, cu, n_seqs,
                                    _ptr_array(gathered), len(gathered), _ptr(st), _stream(dev)))


def sp_reduce_scatter_seq(partials, shards, *, cu_seqlens=None, status=None):
    """g* alone: shards[k] = bf16(sum_r partials[r][:, o_k:o_{k+1}, :])."""
    lib = load()
    t = len(partials)
    b, s, h = partials[0].shape
    dev = partials[0].device
    sizes = shard_sizes(s, t)
    for r in range(t):
        _need(partials[r], (b, s, h), torch.bfloat16, dev, f"partials[{r}]")
        _need(shards[r], (b, sizes[r], h), torch.bfloat16, dev, f"shards[{r}]")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        _check(lib.sp_reduce_scatter_seq(_ptr_array(partials), b, s, h, t, cu, n_seqs,
                                         _ptr_array(shards), _ptr(st), _stream(dev)))


def sp_norm_bwd_workspace_bytes(b, s, h, t, norm="layernorm"):
    return int(load().sp_norm_bwd_workspace_bytes(b, s, h, t, NORMS[norm]))


def sp_norm_bwd(dy, z, mask, mean, rstd, gamma, dz_skip=None, *, s, p, cu_seqlens=None,
                norm="layernorm", dresidual, dgathered, dgamma=None, dbeta=None, dbias=None,
                workspace, status=None):
    """Backward of the boundary (writes the given outputs)."""
    _norm_bwd_call("sp_norm_bwd", 1, dy, z, mask, mean, rstd, gamma, dz_skip, s, p,
                   cu_seqlens, norm, dresidual, dgathered, dgamma, dbeta, dbias, workspace,
                   status)


def sp_norm_bwd_bitmask(dy, z, mask_bits, mean, rstd, gamma, dz_skip=None, *, s, p,
                        cu_seqlens=None, norm="layernorm", dresidual, dgathered, dgamma=None,
                        dbeta=None, dbias=None, workspace, status=None):
    """sp_norm_bwd reading the mask stored one bit per element
    (mask_bits[k]: (b, s_k, h / 8) uint8, bit e of byte j = channel 8j + e)."""
    _norm_bwd_call("sp_norm_bwd_bitmask", 8, dy, z, mask_bits, mean, rstd, gamma, dz_skip, s,
                   p, cu_seqlens, norm, dresidual, dgathered, dgamma, dbeta, dbias, workspace,
                   status)


def _norm_bwd_call(entry, mask_div, dy, z, mask, mean, rstd, gamma, dz_skip, s, p, cu_seqlens,
                   norm, dresidual, dgathered, dgamma, dbeta, dbias, workspace, status):
    lib = load()
    t = len(dy)
    b, _, h = dy[0].shape
    dev = dy[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    ln = norm == "layernorm"
    for k in range(t):
        _need(dy[k], (b, sizes[k], h), bf, dev, f"dy[{k}]")
        _need(z[k], (b, sizes[k], h), bf, dev, f"z[{k}]")
        _need(mask[k], (b, sizes[k], h // mask_div), torch.uint8, dev, f"mask[{k}]")
        _need(rstd[k], (b, sizes[k]), torch.float32, dev, f"rstd[{k}]")
        if ln:
            _need(mean[k], (b, sizes[k]), torch.float32, dev, f"mean[{k}]")
        if dz_skip is not None:
            _need(dz_skip[k], (b, sizes[k], h), bf, dev, f"dz_skip[{k}]")
        _need(dresidual[k], (b, sizes[k], h), bf, dev, f"dresidual[{k}]")
    for j, g in enumerate(dgathered):
        _need(g, (b, s, h), bf, dev, f"dgathered[{j}]")
    _need(gamma, (h,), bf, dev, "gamma")
    for name, v in (("dgamma", dgamma), ("dbeta", dbeta), ("dbias", dbias)):
        if v is not None:
            _need(v, (h,), torch.float32, dev, name)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        code = getattr(lib, entry)(
            _ptr_array(dy), _ptr_array(z), _ptr_array(mask), _ptr_array(mean) if ln else None,
            _ptr_array(rstd), _ptr(gamma), _ptr_array(dz_skip), b, s, h, t, float(p), cu, n_seqs,
            NORMS[norm], _ptr_array(dresidual), _ptr_array(dgathered), len(dgathered),
            _ptr(dgamma), _ptr(dbeta) if ln else None, _ptr(dbias), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(st), _stream(dev))
    _check(code)


def sp_rs_norm_bwd(dy_partials, z, mask, mean, rstd, gamma, dz_skip=None, *, p,
                   cu_seqlens=None, norm="layernorm", dresidual, dgathered, dgamma=None,
                   dbeta=None, dbias=None, workspace, status=None):
    """Backward entered through g: reduce-scatter of the t partial gradients of
    the gathered input, fused into the norm / dropout backward."""
    _rs_norm_bwd_call("sp_rs_norm_bwd", 1, dy_partials, z, mask, mean, rstd, gamma, dz_skip, p,
                      cu_seqlens, norm, dresidual, dgathered, dgamma, dbeta, dbias, workspace,
                      status)


def sp_rs_norm_bwd_bitmask(dy_partials, z, mask_bits, mean, rstd, gamma, dz_skip=None, *, p,
                           cu_seqlens=None, norm="layernorm", dresidual, dgathered,
                           dgamma=None, dbeta=None, dbias=None, workspace, status=None):
    """sp_rs_norm_bwd reading the mask stored one bit per element
    (mask_bits[k]: (b, s_k, h / 8) uint8, bit e of byte j = channel 8j + e)."""
    _rs_norm_bwd_call("sp_rs_norm_bwd_bitmask", 8, dy_partials, z, mask_bits, mean, rstd, gamma,
                      dz_skip, p, cu_seqlens, norm, dresidual, dgathered, dgamma, dbeta, dbias,
                      workspace, status)


def _rs_norm_bwd_call(entry, mask_div, dy_partials, z, mask, mean, rstd, gamma, dz_skip, p,
                      cu_seqlens, norm, dresidual, dgathered, dgamma, dbeta, dbias, workspace,
                      status):
    lib = load()
    t = len(dy_partials)
    b, s, h = dy_partials[0].shape
    dev = dy_partials[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    ln = norm == "layernorm"
    for r in range(t):
        _need(dy_partials[r], (b, s, h), bf, dev, f"dy_partials[{r}]")
    for k in range(t):
        _need(z[k], (b, sizes[k], h), bf, dev, f"z[{k}]")
        _need(mask[k], (b, sizes[k], h // mask_div), torch.uint8, dev, f"mask[{k}]")
        _need(rstd[k], (b, sizes[k]), torch.float32, dev, f"rstd[{k}]")
        if ln:
            _need(mean[k], (b, sizes[k]), torch.float32, dev, f"mean[{k}]")
        if dz_skip is not None:
            _need(dz_skip[k], (b, sizes[k], h), bf, dev, f"dz_skip[{k}]")
        _need(dresidual[k], (b, sizes[k], h), bf, dev, f"dresidual[{k}]")
    for j, g in enumerate(dgathered):
        _need(g, (b, s, h), bf, dev, f"dgathered[{j}]")
    _need(gamma, (h,), bf, dev, "gamma")
    for name, v in (("dgamma", dgamma), ("dbeta", dbeta), ("dbias", dbias)):
        if v is not None:
            _need(v, (h,), torch.float32, dev, name)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        _check(getattr(lib, entry)(
            _ptr_array(dy_partials), _ptr_array(z), _ptr_array(mask),
            _ptr_array(mean) if ln else None, _ptr_array(rstd), _ptr(gamma), _ptr_array(dz_skip),
            b, s, h, t, float(p), cu, n_seqs, NORMS[norm], _ptr_array(dresidual),
            _ptr_array(dgathered), len(dgathered), _ptr(dgamma), _ptr(dbeta) if ln else None,
            _ptr(dbias), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(st),
            _stream(dev)))


def sp_norm_bwd_philox(dy, z, mean, rstd, gamma, dz_skip=None, *, s, p, seed, offset=0,
                       cu_seqlens=None, norm="layernorm", dresidual, dgathered, dgamma=None,
                       dbeta=None, dbias=None, workspace, status=None):
    """Mask-free backward: the dropout mask is drawn again from (seed, offset, p)."""
    lib = load()
    t = len(dy)
    b, _, h = dy[0].shape
    dev = dy[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    ln = norm == "layernorm"
    for k in range(t):
        _need(dy[k], (b, sizes[k], h), bf, dev, f"dy[{k}]")
        _need(z[k], (b, sizes[k], h), bf, dev, f"z[{k}]")
        _need(rstd[k], (b, sizes[k]), torch.float32, dev, f"rstd[{k}]")
        if ln:
            _need(mean[k], (b, sizes[k]), torch.float32, dev, f"mean[{k}]")
        if dz_skip is not None:
            _need(dz_skip[k], (b, sizes[k], h), bf, dev, f"dz_skip[{k}]")
        _need(dresidual[k], (b, sizes[k], h), bf, dev, f"dresidual[{k}]")
    for j, g in enumerate(dgathered):
        _need(g, (b, s, h), bf, dev, f"dgathered[{j}]")
    _need(gamma, (h,), bf, dev, "gamma")
    for name, v in (("dgamma", dgamma), ("dbeta", dbeta), ("dbias", dbias)):
        if v is not None:
            _need(v, (h,), torch.float32, dev, name)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        _check(lib.sp_norm_bwd_philox(
            _ptr_array(dy), _ptr_array(z), _ptr_array(mean) if ln else None, _ptr_array(rstd),
            _ptr(gamma), _ptr_array(dz_skip), b, s, h, t, float(p), int(seed), int(offset), cu,
            n_seqs, NORMS[norm], _ptr_array(dresidual), _ptr_array(dgathered), len(dgathered),
            _ptr(dgamma), _ptr(dbeta) if ln else None, _ptr(dbias), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(st), _stream(dev)))


NOALLOC_WORKSPACE_BYTES = 16 << 20


def sp_norm_bwd_noalloc(dy, z, mask, mean, rstd, gamma, dz_skip=None, *, s, p, cu_seqlens=None,
                        norm="layernorm", dresidual, dgathered, dgamma=None, dbeta=None,
                        dbias=None, status=None):
    """sp_norm_bwd for callers that cannot allocate: no workspace argument.

    The library keeps the parameter-gradient partials in a fixed array of its
    own device memory (16 MiB per GPU, for the life of the process), so a
    caller that has no allocator to draw scratch from can still run the
    backward.  Calls on one device share that array: do not let two of them
    run concurrently on different streams.  The first call on a device looks
    up the array's address; make it before any stream capture.
    """
    lib = load()
    t = len(dy)
    b, _, h = dy[0].shape
    dev = dy[0].device
    bf = torch.bfloat16
    sizes = shard_sizes(s, t)
    ln = norm == "layernorm"
    for k in range(t):
        _need(dy[k], (b, sizes[k], h), bf, dev, f"dy[{k}]")
        _need(z[k], (b, sizes[k], h), bf, dev, f"z[{k}]")
        _need(mask[k], (b, sizes[k], h), torch.uint8, dev, f"mask[{k}]")
        _need(rstd[k], (b, sizes[k]), torch.float32, dev, f"rstd[{k}]")
        if ln:
            _need(mean[k], (b, sizes[k]), torch.float32, dev, f"mean[{k}]")
        if dz_skip is not None:
            _need(dz_skip[k], (b, sizes[k], h), bf, dev, f"dz_skip[{k}]")
        _need(dresidual[k], (b, sizes[k], h), bf, dev, f"dresidual[{k}]")
    for j, g in enumerate(dgathered):
        _need(g, (b, s, h), bf, dev, f"dgathered[{j}]")
    _need(gamma, (h,), bf, dev, "gamma")
    for name, v in (("dgamma", dgamma), ("dbeta", dbeta), ("dbias", dbias)):
        if v is not None:
            _need(v, (h,), torch.float32, dev, name)
    cu, n_seqs = _seq_meta(cu_seqlens, b, dev)
    st = device_status(dev) if status is None else status
    with _on_device(dev):
        code = lib.sp_norm_bwd_noalloc(
            _ptr_array(dy), _ptr_array(z), _ptr_array(mask), _ptr_array(mean) if ln else None,
            _ptr_array(rstd), _ptr(gamma), _ptr_array(dz_skip), b, s, h, t, float(p), cu, n_seqs,
            NORMS[norm], _ptr_array(dresidual), _ptr_array(dgathered), len(dgathered),
            _ptr(dgamma), _ptr(dbeta) if ln else None, _ptr(dbias), _ptr(st), _stream(dev))
    _check(code)


def sp_debug_inject(code):
    load().sp_debug_inject(int(code))


def sp_debug_tune(kernel, stages=0, blocks_per_sm=0, threads=0, chunks=0):
    _check(load().sp_debug_tune(int(kernel), int(stages), int(blocks_per_sm), int(threads),
                                int(chunks)))


def sp_debug_last_shape(kernel):
    """Launch shape of this thread's last forward (0) or backward (1) call:
    dict(threads, chunks, stages, grid, cluster, smem)."""
    out = (ctypes.c_int32 * 6)()
    _check(load().sp_debug_last_shape(int(kernel), ctypes.cast(out, _vp)))
    return dict(zip(("threads", "chunks", "stages", "grid", "cluster", "smem"), list(out)))


def sp_debug_philox(ctr_key):
    """Device Philox4x32-10 of an (n, 6) uint32 tensor of (c0..c3, k0, k1)."""
    if ctr_key.dtype != torch.int32 or ctr_key.dim() != 2 or ctr_key.shape[1] != 6:
        raise ValueError("ctr_key must be an (n, 6) int32 tensor (uint32 bits)")
    out = torch.empty((ctr_key.shape[0], 4), dtype=torch.int32, device=ctr_key.device)
    _check(load().sp_debug_philox(_ptr(ctr_key.contiguous()), _ptr(out), ctr_key.shape[0],
                                  _stream(ctr_key.device)))
    return out


def sp_abi_version():
    return int(load().sp_abi_version())
