"""ctypes binding of ``libpoetx.so`` (the C ABI declared in ``include/poetx.h``).

Argument marshalling only: every function takes torch tensors, passes their
device pointers and the current CUDA stream to the C entry point of the same
name, and raises ``PoetxError`` on a non-OK status.  No step of the layer runs
in Python and there is no fallback: if the library is missing, loading fails
with an error that says how to build it.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpoetx.so")

F32, BF16 = 0, 1
STATUS = {0: "POETX_OK", 1: "POETX_ERR_INVALID_ARG", 2: "POETX_ERR_SHAPE",
          3: "POETX_ERR_UNSUPPORTED", 4: "POETX_ERR_NOT_PERMUTATION", 5: "POETX_ERR_CUDA",
          6: "POETX_ERR_TIMEOUT", 7: "POETX_ERR_RANGE"}

# every symbol include/poetx.h declares
EXPORTS = ["poetx_status_string", "poetx_version", "poetx_cayley_neumann",
           "poetx_cayley_neumann_pair",
           "poetx_cayley_neumann_backward", "poetx_invert_perm", "poetx_check_perm",
           "poetx_merge_w0", "poetx_workspace_bytes", "poetx_forward", "poetx_backward",
           "poetx_stream_status", "poetx_launch_count", "poetx_profile_enable",
           "poetx_profile_report", "poetx_forward_noalloc", "poetx_fold_workspace_bytes",
           "poetx_fold_w0", "poetx_quantize_w0", "poetx_dequantize_w0",
           "poetx_workspace_bytes_xq", "poetx_forward_xq", "poetx_backward_xq",
           "poetx_diag_expire_wait"]


class PoetxError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s" % (fn, STATUS.get(code, code)))
        self.code = code


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libpoetx.so not found at %s: build it with "
                          "`python -m orthogonal_equivalence_neumann_b300.build`" % path)
    lib = ctypes.CDLL(path)
    P, I, Z, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
    sig = {
        "poetx_status_string": (ctypes.c_char_p, [I]),
        "poetx_version": (I, []),
        "poetx_cayley_neumann": (I, [P, I, I, I, P, I, P]),
        "poetx_cayley_neumann_pair": (I, [P, I, I, P, I, I, I, P, P, I, P]),
        "poetx_cayley_neumann_backward": (I, [P, P, I, I, I, P, P]),
        "poetx_invert_perm": (I, [P, P, I, P]),
        "poetx_check_perm": (I, [P, P, I, P, P]),
        "poetx_merge_w0": (I, [P, P, I, I, I, P, P, P]),
        "poetx_workspace_bytes": (Z, [I, I, I, I, I, I]),
        "poetx_forward": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, Z, P]),
        "poetx_backward": (I, [P, P, P, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P,
                               P, Z, P]),
        "poetx_stream_status": (I, [P]),
        "poetx_diag_expire_wait": (I, [I, U, P]),
        "poetx_forward_noalloc": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]),
        "poetx_launch_count": (ctypes.c_ulonglong, []),
        "poetx_profile_enable": (I, [I]),
        "poetx_profile_report": (I, [ctypes.c_char_p, Z]),
        "poetx_fold_workspace_bytes": (Z, [I, I, I, I, I]),
        "poetx_fold_w0": (I, [P, P, P, P, P, I, I, I, I, I, P, P, Z, P]),
        "poetx_quantize_w0": (I, [P, I, I, I, P, P, P]),
        "poetx_dequantize_w0": (I, [P, P, I, I, I, P, P]),
        "poetx_workspace_bytes_xq": (Z, [I, I, I, I, I, I]),
        "poetx_forward_xq": (I, [P] * 9 + [I] * 6 + [P, P, P, Z, P]),
        "poetx_backward_xq": (I, [P] * 6 + [I] + [P] * 7 + [I] * 6 + [P] * 4 + [Z, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(dt) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise TypeError("unsupported dtype %s" % dt)


def _check(name, code):
    if code != 0:
        raise PoetxError(name, code)


def poetx_version() -> int:
    return load().poetx_version()


def poetx_status_string(code: int) -> str:
    return load().poetx_status_string(code).decode()


def poetx_cayley_neumann(theta, b, n, Q, stream=None):
    """Q [nb, b, b] (fp32 or bf16) <- Cayley-Neumann blocks of theta [nb, b(b-1)/2] fp32."""
    nb = theta.shape[0]
    _check("poetx_cayley_neumann", load().poetx_cayley_neumann(
        _ptr(theta), nb, b, n, _ptr(Q), dtype_code(Q.dtype), _stream(stream)))


def poetx_cayley_neumann_pair(theta_P, b_P, theta_R, b_R, n, Q_P, Q_R, stream=None):
    """Both factors of a layer in one call (Q_P and Q_R share a dtype)."""
    if Q_P.dtype != Q_R.dtype:
        raise TypeError("Q_P and Q_R must share a dtype")
    _check("poetx_cayley_neumann_pair", load().poetx_cayley_neumann_pair(
        _ptr(theta_P), theta_P.shape[0], b_P, _ptr(theta_R), theta_R.shape[0], b_R, n,
        _ptr(Q_P), _ptr(Q_R), dtype_code(Q_P.dtype), _stream(stream)))


def poetx_cayley_neumann_backward(theta, dQ, b, n, dtheta, stream=None):
    nb = theta.shape[0]
    _check("poetx_cayley_neumann_backward", load().poetx_cayley_neumann_backward(
        _ptr(theta), _ptr(dQ), nb, b, n, _ptr(dtheta), _stream(stream)))


def poetx_invert_perm(perm, inv, stream=None):
    _check("poetx_invert_perm", load().poetx_invert_perm(_ptr(perm), _ptr(inv), perm.numel(),
                                                         _stream(stream)))


def poetx_check_perm(perm, inv, scratch, stream=None) -> int:
    """Returns the status code (0 = valid permutation, 4 = not a permutation)."""
    code = load().poetx_check_perm(_ptr(perm), _ptr(inv), perm.numel(), _ptr(scratch),
                                   _stream(stream))
    if code not in (0, 4):
        raise PoetxError("poetx_check_perm", code)
    return code


def poetx_merge_w0(W0, W0m, perm_out, perm_in, stream=None):
    d_out, d_in = W0.shape
    _check("poetx_merge_w0", load().poetx_merge_w0(
        _ptr(W0), _ptr(W0m), d_out, d_in, dtype_code(W0.dtype), _ptr(perm_out), _ptr(perm_in),
        _stream(stream)))


def poetx_fold_workspace_bytes(d_out, d_in, b_in, b_out, dtype) -> int:
    return int(load().poetx_fold_workspace_bytes(d_out, d_in, b_in, b_out, dtype_code(dtype)))


def poetx_fold_w0(W0m, Q_P, Q_R, perm_in, perm_out, b_in, b_out, W0_new, workspace, stream=None):
    d_out, d_in = W0m.shape
    _check("poetx_fold_w0", load().poetx_fold_w0(
        _ptr(W0m), _ptr(Q_P), _ptr(Q_R), _ptr(perm_in), _ptr(perm_out), d_out, d_in, b_in, b_out,
        dtype_code(W0m.dtype), _ptr(W0_new), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def poetx_workspace_bytes(T, d_in, d_out, b_in, b_out, dtype) -> int:
    return int(load().poetx_workspace_bytes(T, d_in, d_out, b_in, b_out, dtype_code(dtype)))


def poetx_forward(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, b_in, b_out, y, z_save,
                  workspace, stream=None):
    T, d_in = x.shape
    d_out = W0m.shape[0]
    _check("poetx_forward", load().poetx_forward(
        _ptr(x), _ptr(W0m), _ptr(Q_P), _ptr(Q_R), _ptr(perm_in), _ptr(inv_in), _ptr(perm_out),
        _ptr(inv_out), T, d_in, d_out, b_in, b_out, dtype_code(x.dtype), _ptr(y), _ptr(z_save),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def poetx_backward(x, dy, W0m, theta_P, theta_R, n, Q_P, Q_R, z_saved, perm_in, inv_in, perm_out,
                   inv_out, b_in, b_out, dX, dtheta_P, dtheta_R, workspace, stream=None):
    T, d_in = x.shape
    d_out = W0m.shape[0]
    _check("poetx_backward", load().poetx_backward(
        _ptr(x), _ptr(dy), _ptr(W0m), _ptr(theta_P), _ptr(theta_R), n, _ptr(Q_P), _ptr(Q_R),
        _ptr(z_saved), _ptr(perm_in), _ptr(inv_in), _ptr(perm_out), _ptr(inv_out), T, d_in, d_out,
        b_in, b_out, dtype_code(x.dtype), _ptr(dX), _ptr(dtheta_P), _ptr(dtheta_R),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def poetx_forward_noalloc(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, b_in, b_out, y,
                          z_save, stream=None):
    """poetx_forward with the library's static device workspace (no allocation)."""
    T, d_in = x.shape
    d_out = W0m.shape[0]
    _check("poetx_forward_noalloc", load().poetx_forward_noalloc(
        _ptr(x), _ptr(W0m), _ptr(Q_P), _ptr(Q_R), _ptr(perm_in), _ptr(inv_in), _ptr(perm_out),
        _ptr(inv_out), T, d_in, d_out, b_in, b_out, dtype_code(x.dtype), _ptr(y), _ptr(z_save),
        _stream(stream)))


def poetx_quantize_w0(W0, W0q, scale, stream=None):
    d_out, d_in = W0.shape
    _check("poetx_quantize_w0", load().poetx_quantize_w0(
        _ptr(W0), d_out, d_in, dtype_code(W0.dtype), _ptr(W0q), _ptr(scale), _stream(stream)))


def poetx_dequantize_w0(W0q, scale, W0, stream=None):
    d_out, d_in = W0q.shape
    _check("poetx_dequantize_w0", load().poetx_dequantize_w0(
        _ptr(W0q), _ptr(scale), d_out, d_in, dtype_code(W0.dtype), _ptr(W0), _stream(stream)))


def poetx_workspace_bytes_xq(T, d_in, d_out, b_in, b_out, dtype) -> int:
    return int(load().poetx_workspace_bytes_xq(T, d_in, d_out, b_in, b_out, dtype_code(dtype)))


def poetx_forward_xq(x, W0q, scale, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, b_in, b_out, y,
                     z_save, workspace, stream=None):
    T, d_in = x.shape
    d_out = W0q.shape[0]
    _check("poetx_forward_xq", load().poetx_forward_xq(
        _ptr(x), _ptr(W0q), _ptr(scale), _ptr(Q_P), _ptr(Q_R), _ptr(perm_in), _ptr(inv_in),
        _ptr(perm_out), _ptr(inv_out), T, d_in, d_out, b_in, b_out, dtype_code(x.dtype), _ptr(y),
        _ptr(z_save), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def poetx_backward_xq(x, dy, W0q, scale, theta_P, theta_R, n, Q_P, Q_R, z_saved, perm_in, inv_in,
                      perm_out, inv_out, b_in, b_out, dX, dtheta_P, dtheta_R, workspace,
                      stream=None):
    T, d_in = x.shape
    d_out = W0q.shape[0]
    _check("poetx_backward_xq", load().poetx_backward_xq(
        _ptr(x), _ptr(dy), _ptr(W0q), _ptr(scale), _ptr(theta_P), _ptr(theta_R), n, _ptr(Q_P),
        _ptr(Q_R), _ptr(z_saved), _ptr(perm_in), _ptr(inv_in), _ptr(perm_out), _ptr(inv_out), T,
        d_in, d_out, b_in, b_out, dtype_code(x.dtype), _ptr(dX), _ptr(dtheta_P), _ptr(dtheta_R),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def poetx_stream_status(stream=None):
    _check("poetx_stream_status", load().poetx_stream_status(_stream(stream)))


def poetx_diag_expire_wait(cluster_scope: int, polls: int, stream=None):
    """Launch one bounded device wait that runs out (the failure path's check)."""
    _check("poetx_diag_expire_wait", load().poetx_diag_expire_wait(cluster_scope, polls,
                                                                   _stream(stream)))


def poetx_launch_count() -> int:
    return int(load().poetx_launch_count())


def poetx_profile_enable(enable: bool):
    load().poetx_profile_enable(1 if enable else 0)


def poetx_profile_report() -> dict:
    """{kernel name: (launches, total_ms)} for the launches recorded since the last report."""
    buf = ctypes.create_string_buffer(1 << 16)
    n = load().poetx_profile_report(buf, len(buf))
    if n < 0:
        raise PoetxError("poetx_profile_report", 5)
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out
