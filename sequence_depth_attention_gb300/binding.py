"""ctypes binding of ``libmoda.so``: the calls of ``include/moda.h`` with the
same names, taking torch CUDA tensors and marshalling their pointers and the
current stream. Every step of the computation runs in the library's kernels;
this module only allocates outputs when the caller does not pass them.

The library is built in-tree (``python -m sequence_depth_attention_gb300.build``
or ``__graft_entry__.build()``) into ``sequence_depth_attention_gb300/_build``.
If it is missing, loading raises ``ModaError``: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "_build", "libmoda.so")

MODA_OK = 0
_STATUS = {0: "MODA_OK", 1: "MODA_ERR_INVALID_ARG", 2: "MODA_ERR_UNSUPPORTED",
           3: "MODA_ERR_MISALIGNED", 4: "MODA_ERR_CUDA", 5: "MODA_ERR_TIMEOUT",
           6: "MODA_ERR_NO_DEVICE"}

# every symbol include/moda.h declares
EXPORTS = ("moda_pack_depth", "moda_depth_write", "moda_depth_write_at", "moda_depth_mass",
           "moda_depth_mass_workspace_bytes", "moda_depth_cache_admit", "moda_kv_proj_write",
           "moda_fwd", "moda_fwd_layer_major", "moda_fwd_layer_major_host",
           "moda_fwd_host_workspace_bytes", "moda_fwd_depth_cc", "moda_decode",
           "moda_decode_strided",
           "moda_decode_workspace_bytes", "moda_bwd", "moda_bwd_layer_major", "moda_bwd_noalloc", "moda_get_device_error",
           "moda_selftest_wait_timeout", "moda_status_string", "moda_last_error_detail")

_lock = threading.Lock()
_lib = None


class ModaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = _STATUS.get(status, f"status {status}")
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


def library_path() -> str:
    return _LIB


def load():
    """Load libmoda.so once; raises ModaError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB):
            raise ModaError(6, "load", f"{_LIB} is missing; build it with "
                            "`python -m sequence_depth_attention_gb300.build`")
        lib = ctypes.CDLL(_LIB)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.moda_pack_depth.argtypes = [vp, vp, i, i, i, i, vp]
        lib.moda_pack_depth.restype = i
        lib.moda_depth_write.argtypes = [vp, vp, i, i, i, i, i, vp]
        lib.moda_kv_proj_write.restype = i
        lib.moda_kv_proj_write.argtypes = [vp, vp, vp] + [i] * 6 + [vp, vp, vp]
        lib.moda_depth_write.restype = i
        lib.moda_depth_write_at.argtypes = [vp, vp, i, i, i, i, vp, vp]
        lib.moda_depth_write_at.restype = i
        lib.moda_depth_mass_workspace_bytes.argtypes = [i, i, i]
        lib.moda_depth_mass_workspace_bytes.restype = ctypes.c_size_t
        lib.moda_depth_mass.argtypes = [vp, vp, vp] + [i] * 5 + [f, vp, vp, ctypes.c_size_t, vp]
        lib.moda_depth_mass.restype = i
        lib.moda_depth_cache_admit.argtypes = [vp, vp, i, i, i, i, vp, vp]
        lib.moda_depth_cache_admit.restype = i
        lib.moda_decode_workspace_bytes.argtypes = [i, i, i]
        lib.moda_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.moda_decode.argtypes = [vp] * 5 + [ctypes.c_longlong] + [i] * 5 + [f, vp, vp, vp,
                                                                           ctypes.c_size_t, vp]
        lib.moda_decode.restype = i
        lib.moda_decode_strided.argtypes = [vp] * 5 + [ctypes.c_longlong] * 2 + [i] * 5 + [
            f, vp, vp, vp, ctypes.c_size_t, vp]
        lib.moda_decode_strided.restype = i
        lib.moda_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, vp]
        lib.moda_fwd_depth_cc.restype = i
        lib.moda_fwd_depth_cc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, vp]
        lib.moda_fwd.restype = i
        lib.moda_fwd_layer_major.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, vp]
        lib.moda_fwd_layer_major.restype = i
        lib.moda_fwd_host_workspace_bytes.argtypes = [i] * 5
        lib.moda_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.moda_fwd_layer_major_host.argtypes = [vp] * 5 + [i] * 5 + [f, vp, vp, vp,
                                                                        ctypes.c_size_t, vp]
        lib.moda_fwd_layer_major_host.restype = i
        lib.moda_bwd.argtypes = [vp] * 8 + [i] * 5 + [f] + [vp] * 7
        lib.moda_bwd_layer_major.argtypes = [vp] * 8 + [i] * 5 + [f] + [vp] * 7
        lib.moda_bwd_layer_major.restype = i
        lib.moda_bwd.restype = i
        lib.moda_bwd_noalloc.argtypes = [vp] * 8 + [i] * 5 + [f] + [vp] * 6
        lib.moda_bwd_noalloc.restype = i
        lib.moda_get_device_error.argtypes = [vp]
        lib.moda_get_device_error.restype = i
        lib.moda_selftest_wait_timeout.argtypes = [i, vp]
        lib.moda_selftest_wait_timeout.restype = i
        lib.moda_status_string.argtypes = [i]
        lib.moda_status_string.restype = ctypes.c_char_p
        lib.moda_last_error_detail.argtypes = []
        lib.moda_last_error_detail.restype = ctypes.c_char_p
        _lib = lib
        return lib


def moda_status_string(status: int) -> str:
    return load().moda_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MODA_OK:
        detail = load().moda_last_error_detail().decode()
        raise ModaError(status, where, detail)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def moda_pack_depth(src: torch.Tensor, dst: torch.Tensor | None = None, stream=None):
    """[L,T,Hk,d] -> [Hk,T,L,d] (bit-exact). Returns dst.

    src may be a CUDA tensor or a pinned (page-locked) CPU tensor; the kernel
    then reads it over the host link, so the transfer and the relayout are one
    pass. dst is always a CUDA tensor."""
    if src.is_cuda:
        _need(src, "src")
    else:
        if not isinstance(src, torch.Tensor) or src.dtype != torch.bfloat16 or not src.is_contiguous():
            raise TypeError("src: expected a contiguous bf16 tensor")
        if not src.is_pinned():
            raise ValueError("src: a CPU tensor must be pinned (page-locked)")
    L, T, Hk, d = src.shape
    if dst is None:
        dev = src.device if src.is_cuda else torch.device("cuda", torch.cuda.current_device())
        dst = torch.empty((Hk, T, L, d), dtype=src.dtype, device=dev)
    _need(dst, "dst")
    if tuple(dst.shape) != (Hk, T, L, d):
        raise ValueError(f"dst: expected shape {(Hk, T, L, d)}, got {tuple(dst.shape)}")
    st = load().moda_pack_depth(_ptr(src), _ptr(dst), L, T, Hk, d, _stream(stream))
    _check(st, "moda_pack_depth")
    return dst


def moda_depth_write(src: torch.Tensor, dst: torch.Tensor, slot: int, stream=None):
    """Write one layer's K or V src[T,Hk,d] into slot `slot` of the packed
    depth stream dst[Hk,T,L,d] (bit-exact). Returns dst."""
    _need(src, "src"), _need(dst, "dst")
    T, Hk, d = src.shape
    if dst.dim() != 4 or dst.shape[0] != Hk or dst.shape[1] != T or dst.shape[3] != d:
        raise ValueError(f"dst must be [Hk,T,L,d] with Hk={Hk}, T={T}, d={d}")
    L = dst.shape[2]
    st = load().moda_depth_write(_ptr(src), _ptr(dst), T, Hk, d, L, int(slot), _stream(stream))
    _check(st, "moda_depth_write")
    return dst


def moda_depth_write_at(src: torch.Tensor, dst: torch.Tensor, slot: torch.Tensor, stream=None):
    """dst[:, :, slot[0], :] = src permuted, with the slot index read from the
    int32 device tensor `slot` when the kernel runs."""
    _need(src, "src"), _need(dst, "dst")
    _need(slot, "slot", torch.int32)
    Hk, T, L, d = dst.shape
    if tuple(src.shape) != (T, Hk, d):
        raise ValueError(f"src must be [T,Hk,d] = {(T, Hk, d)}")
    st = load().moda_depth_write_at(_ptr(src), _ptr(dst), T, Hk, d, L, _ptr(slot),
                                    _stream(stream))
    _check(st, "moda_depth_write_at")
    return dst


def moda_depth_mass_workspace_bytes(T: int, Hk: int, L: int) -> int:
    return int(load().moda_depth_mass_workspace_bytes(int(T), int(Hk), int(L)))


def moda_depth_mass(q, kd, lse, scale: float, mass=None, workspace=None, stream=None):
    """Probability mass [Hk, L] (fp32) that the joint softmax of moda_fwd gives
    each depth slot, summed over the rows of each KV head; lse is the one
    moda_fwd returned for q and kd (packed [Hk,T,L,d])."""
    _need(q, "q"), _need(kd, "kd")
    _need(lse, "lse", torch.float32)
    T, Hq, d = q.shape
    Hk, _, L, _ = kd.shape
    if mass is None:
        mass = torch.empty((Hk, L), dtype=torch.float32, device=q.device)
    _need(mass, "mass", torch.float32)
    nbytes = moda_depth_mass_workspace_bytes(T, Hk, L)
    if workspace is None:
        workspace = torch.empty(((nbytes + 3) // 4,), dtype=torch.float32, device=q.device)
    _need(workspace, "workspace", torch.float32)
    st = load().moda_depth_mass(_ptr(q), _ptr(kd), _ptr(lse), T, Hq, Hk, d, L, float(scale),
                                _ptr(mass), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "moda_depth_mass")
    return mass


def moda_depth_cache_admit(slot_age: torch.Tensor, mass: torch.Tensor, recent: int, new_age: int,
                           slot=None, stream=None):
    """Chooses the slot for the entry of age new_age (bounded depth cache) and
    records it in slot_age (int32 [S], -1 = empty); mass is [Hk, S] fp32.
    Returns the int32 device tensor holding the slot."""
    _need(slot_age, "slot_age", torch.int32)
    _need(mass, "mass", torch.float32)
    S = slot_age.shape[0]
    Hk = mass.shape[0]
    if tuple(mass.shape) != (Hk, S):
        raise ValueError(f"mass must be [Hk, S] with S = {S}")
    if slot is None:
        slot = torch.empty((1,), dtype=torch.int32, device=slot_age.device)
    _need(slot, "slot", torch.int32)
    st = load().moda_depth_cache_admit(_ptr(slot_age), _ptr(mass), Hk, S, int(recent),
                                       int(new_age), _ptr(slot), _stream(stream))
    _check(st, "moda_depth_cache_admit")
    return slot


def moda_kv_proj_write(x: torch.Tensor, wk: torch.Tensor, wv: torch.Tensor, kd: torch.Tensor,
                       vd: torch.Tensor, slot: int, stream=None):
    """An FFN layer's depth pair: K = x wk^T and V = x wv^T (bf16, fp32
    accumulation) written into slot `slot` of the packed streams kd, vd
    [Hk,T,L,d]. x is [T,Dm]; wk, wv are [Hk*d,Dm]. Returns (kd, vd)."""
    for t, n in ((x, "x"), (wk, "wk"), (wv, "wv"), (kd, "kd"), (vd, "vd")):
        _need(t, n)
    T, Dm = x.shape
    if kd.dim() != 4 or tuple(vd.shape) != tuple(kd.shape) or kd.shape[1] != T:
        raise ValueError(f"kd and vd must both be [Hk,T,L,d] with T={T}")
    Hk, _, L, d = kd.shape
    if tuple(wk.shape) != (Hk * d, Dm) or tuple(wv.shape) != (Hk * d, Dm):
        raise ValueError(f"wk and wv must be [{Hk * d},{Dm}]")
    st = load().moda_kv_proj_write(_ptr(x), _ptr(wk), _ptr(wv), T, Dm, Hk, d, L, int(slot),
                                   _ptr(kd), _ptr(vd), _stream(stream))
    _check(st, "moda_kv_proj_write")
    return kd, vd


def moda_fwd(q, k, v, kd, vd, scale: float, o=None, lse=None, stream=None,
             want_lse: bool = True, depth_on_cuda_cores: bool = False):
    """MoDA forward. q[T,Hq,d], k/v[T,Hk,d], kd/vd packed [Hk,T,L,d] (or
    None when L == 0). Returns (o[T,Hq,d] bf16, lse[T,Hq] fp32 or None).
    depth_on_cuda_cores=True calls moda_fwd_depth_cc (same result, the depth
    slots on CUDA cores in a second pass; lse is then always produced)."""
    if depth_on_cuda_cores:
        want_lse = True
    _need(q, "q"), _need(k, "k"), _need(v, "v")
    T, Hq, d = q.shape
    Hk = k.shape[1]
    if tuple(k.shape) != (T, Hk, d) or tuple(v.shape) != (T, Hk, d):
        raise ValueError("k and v must be [T,Hk,d] matching q[T,Hq,d]")
    if kd is None or kd.numel() == 0:
        L = 0 if kd is None else kd.shape[2]
        if L != 0:
            raise ValueError("empty kd with L > 0")
        kd = vd = None
    else:
        _need(kd, "kd"), _need(vd, "vd")
        L = kd.shape[2]
        if tuple(kd.shape) != (Hk, T, L, d) or tuple(vd.shape) != (Hk, T, L, d):
            raise ValueError(f"kd/vd must be packed [Hk,T,L,d] = {(Hk, T, L, d)}")
    if o is None:
        o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=q.device)
    _need(o, "o")
    if want_lse and lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    fn, name = (load().moda_fwd_depth_cc, "moda_fwd_depth_cc") if depth_on_cuda_cores else \
        (load().moda_fwd, "moda_fwd")
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd), T, Hq, Hk, d, L, float(scale), _ptr(o),
            _ptr(lse), _stream(stream))
    _check(st, name)
    return o, lse


def moda_fwd_layer_major(q, k, v, kd, vd, scale: float, o=None, lse=None, stream=None,
                         want_lse: bool = True):
    """MoDA forward on layer-major depth K/V: kd/vd [L,T,Hk,d] as the layers
    wrote them (or None when L == 0); the forward gathers each depth block
    itself, no relayout pass. Returns (o[T,Hq,d] bf16, lse[T,Hq] fp32 or None)."""
    _need(q, "q"), _need(k, "k"), _need(v, "v")
    T, Hq, d = q.shape
    Hk = k.shape[1]
    if tuple(k.shape) != (T, Hk, d) or tuple(v.shape) != (T, Hk, d):
        raise ValueError("k and v must be [T,Hk,d] matching q[T,Hq,d]")
    if kd is None or kd.numel() == 0:
        L = 0 if kd is None else kd.shape[0]
        if L != 0:
            raise ValueError("empty kd with L > 0")
        kd = vd = None
    else:
        _need(kd, "kd"), _need(vd, "vd")
        L = kd.shape[0]
        if tuple(kd.shape) != (L, T, Hk, d) or tuple(vd.shape) != (L, T, Hk, d):
            raise ValueError(f"kd/vd must be layer-major [L,T,Hk,d] = {(L, T, Hk, d)}")
    if o is None:
        o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=q.device)
    _need(o, "o")
    if want_lse and lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    st = load().moda_fwd_layer_major(_ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd), T, Hq, Hk, d, L,
                                     float(scale), _ptr(o), _ptr(lse), _stream(stream))
    _check(st, "moda_fwd_layer_major")
    return o, lse


def moda_fwd_host_workspace_bytes(T: int, Hq: int, Hk: int, d: int, L: int) -> int:
    return int(load().moda_fwd_host_workspace_bytes(int(T), int(Hq), int(Hk), int(d), int(L)))


def _need_host(t, name, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name}: must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def moda_fwd_layer_major_host(q, k, v, kd, vd, scale: float, o=None, lse=None, workspace=None,
                              device=None, stream=None, want_lse: bool = True):
    """moda_fwd_layer_major from and to host memory: q, k, v, kd, vd are CPU
    tensors (pinned for asynchronous copies; kd/vd [L,T,Hk,d] or None when
    L == 0). The library copies them into `workspace` (a CUDA uint8 tensor of
    at least moda_fwd_host_workspace_bytes bytes; allocated on `device` when
    None), runs the forward there and copies o and lse back into host tensors
    (allocated pinned when None), all on `stream`. Returns (o, lse); they are
    valid once the stream has passed the call."""
    _need_host(q, "q"), _need_host(k, "k"), _need_host(v, "v")
    T, Hq, d = q.shape
    Hk = k.shape[1]
    if tuple(k.shape) != (T, Hk, d) or tuple(v.shape) != (T, Hk, d):
        raise ValueError("k and v must be [T,Hk,d] matching q[T,Hq,d]")
    if kd is None or kd.numel() == 0:
        if kd is not None and kd.shape[0] != 0:
            raise ValueError("empty kd with L > 0")
        L, kd, vd = 0, None, None
    else:
        _need_host(kd, "kd"), _need_host(vd, "vd")
        L = kd.shape[0]
        if tuple(kd.shape) != (L, T, Hk, d) or tuple(vd.shape) != (L, T, Hk, d):
            raise ValueError(f"kd/vd must be layer-major [L,T,Hk,d] = {(L, T, Hk, d)}")
    if o is None:
        o = torch.empty((T, Hq, d), dtype=torch.bfloat16, pin_memory=True)
    _need_host(o, "o")
    if want_lse and lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, pin_memory=True)
    if lse is not None:
        _need_host(lse, "lse", torch.float32)
    need = moda_fwd_host_workspace_bytes(T, Hq, Hk, d, L)
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8)
    st = load().moda_fwd_layer_major_host(_ptr(q), _ptr(k), _ptr(v), _ptr(kd), _ptr(vd), T, Hq, Hk,
                                          d, L, float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
                                          workspace.numel(), _stream(stream))
    _check(st, "moda_fwd_layer_major_host")
    return o, lse


def moda_decode_workspace_bytes(Tctx: int, Hq: int, d: int) -> int:
    return int(load().moda_decode_workspace_bytes(int(Tctx), int(Hq), int(d)))


def moda_decode(q, k_cache, v_cache, kd_tok, vd_tok, scale: float, o=None, lse=None,
                workspace=None, stream=None):
    """One decoding step. q[Hq,d]; k_cache/v_cache[Tctx,Hk,d]; kd_tok/vd_tok
    [Hk,L,d] bf16 views with contiguous rows of d values (e.g. kd_packed[:, t],
    or kd_layer_major[:, t].transpose(0, 1) for [L,T,Hk,d] tensors) or None
    when L == 0. Views whose [L,d] blocks are contiguous go to moda_decode,
    others to moda_decode_strided. Returns (o[Hq,d], lse[Hq])."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    Hq, d = q.shape
    Tctx, Hk, _ = k_cache.shape
    if kd_tok is None or kd_tok.numel() == 0:
        L, stride, slot_stride = 0, 0, 0
        kd_tok = vd_tok = None
    else:
        L = kd_tok.shape[1]
        for t, n in ((kd_tok, "kd_tok"), (vd_tok, "vd_tok")):
            if not t.is_cuda or t.dtype != torch.bfloat16 or t.shape != (Hk, L, d) or \
                    t.stride(2) != 1:
                raise ValueError(f"{n}: expected a bf16 CUDA view [Hk,L,d] with contiguous rows")
        stride = kd_tok.stride(0) if Hk > 1 else L * d  # one head: the stride is never used
        slot_stride = kd_tok.stride(1) if L > 1 else d
        if (Hk > 1 and kd_tok.stride(0) != vd_tok.stride(0)) or \
                (L > 1 and kd_tok.stride(1) != vd_tok.stride(1)):
            raise ValueError("kd_tok and vd_tok must have the same strides")
    if o is None:
        o = torch.empty((Hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((Hq,), dtype=torch.float32, device=q.device)
    need = moda_decode_workspace_bytes(Tctx, Hq, d)
    if workspace is None:
        workspace = torch.empty((need + 3) // 4, dtype=torch.float32, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if slot_stride in (0, d) and (Hk == 1 or stride >= L * d):
        st = load().moda_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kd_tok), _ptr(vd_tok),
                                int(stride), Tctx, Hq, Hk, d, L, float(scale), _ptr(o), _ptr(lse),
                                _ptr(workspace), ws_bytes, _stream(stream))
        _check(st, "moda_decode")
    else:
        st = load().moda_decode_strided(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kd_tok),
                                        _ptr(vd_tok), int(slot_stride), int(stride), Tctx, Hq, Hk,
                                        d, L, float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
                                        ws_bytes, _stream(stream))
        _check(st, "moda_decode_strided")
    return o, lse


def moda_bwd(q, k, v, kd, vd, o, lse, dO, scale: float, grads=None, delta=None, stream=None,
             layer_major: bool = False):
    """Gradients of moda_fwd. Inputs as passed to moda_fwd plus the forward's
    o and lse and the upstream gradient dO[T,Hq,d] (bf16). Returns fp32
    (dq[T,Hq,d], dk[T,Hk,d], dv[T,Hk,d], dkd[Hk,T,L,d], dvd[Hk,T,L,d]) with
    the depth gradients in the packed layout (None when L == 0).
    layer_major=True calls moda_bwd_layer_major: kd/vd as passed to
    moda_fwd_layer_major ([L,T,Hk,d]) and dkd/dvd returned in that layout."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _need(t, n)
    _need(lse, "lse", torch.float32)
    T, Hq, d = q.shape
    Hk = k.shape[1]
    L = 0 if kd is None or kd.numel() == 0 else kd.shape[0 if layer_major else 2]
    if L:
        _need(kd, "kd"), _need(vd, "vd")
    dev = q.device
    dshape = (L, T, Hk, d) if layer_major else (Hk, T, L, d)
    if grads is None:
        f32 = dict(dtype=torch.float32, device=dev)
        grads = (torch.empty((T, Hq, d), **f32), torch.empty((T, Hk, d), **f32),
                 torch.empty((T, Hk, d), **f32),
                 torch.empty(dshape, **f32) if L else None,
                 torch.empty(dshape, **f32) if L else None)
    if delta is None:
        delta = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    dq, dk, dv, dkd, dvd = grads
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv"), (delta, "delta")):
        _need(t, n, torch.float32)
    name = "moda_bwd_layer_major" if layer_major else "moda_bwd"
    st = getattr(load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(kd if L else None),
                               _ptr(vd if L else None), _ptr(o), _ptr(lse), _ptr(dO), T, Hq, Hk,
                               d, L, float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(dkd if L else None), _ptr(dvd if L else None), _ptr(delta),
                               _stream(stream))
    _check(st, name)
    return dq, dk, dv, dkd, dvd


def moda_bwd_noalloc(q, k, v, kd, vd, o, lse, dO, scale: float, grads, stream=None):
    """moda_bwd on the library's fixed scratch (no workspace argument, nothing
    allocated by either side). `grads` = (dq, dk, dv, dkd, dvd) fp32 tensors
    the caller owns (dkd/dvd None when L == 0). T*Hq must be <= 2^20."""
    T, Hq, d = q.shape
    Hk = k.shape[1]
    L = 0 if kd is None or kd.numel() == 0 else kd.shape[2]
    dq, dk, dv, dkd, dvd = grads
    st = load().moda_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kd if L else None),
                                 _ptr(vd if L else None), _ptr(o), _ptr(lse), _ptr(dO), T, Hq, Hk,
                                 d, L, float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(dkd if L else None), _ptr(dvd if L else None),
                                 _stream(stream))
    _check(st, "moda_bwd_noalloc")
    return grads


def moda_get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device's kernel error word."""
    return int(load().moda_get_device_error(_stream(stream)))


def moda_selftest_wait_timeout(timeout_ms: int = 50, stream=None) -> None:
    """Launch the failure-path diagnostic; read its latched status with
    moda_get_device_error()."""
    _check(load().moda_selftest_wait_timeout(int(timeout_ms), _stream(stream)),
           "moda_selftest_wait_timeout")
