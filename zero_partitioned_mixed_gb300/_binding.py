"""ctypes marshalling for libzero_gb300.so (argument conversion only)."""

from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

from .build import LIB_PATH

ZERO_FP16, ZERO_BF16 = 0, 1
ZERO_MODE_AUTO, ZERO_MODE_TWO_PASS_WS, ZERO_MODE_TWO_PASS_REREAD, ZERO_MODE_SPECULATIVE = 0, 1, 2, 3
ZERO_MODE_SPECULATIVE_STAGED = 4
ZERO_F_DOUBLE_BUFFER = 1
ZERO_MAX_RANKS = 64

ZERO_ETIMEOUT = 4
STATUS_NAMES = {0: "ZERO_OK", 1: "ZERO_EINVAL", 2: "ZERO_ENOMEM", 3: "ZERO_ECUDA",
                4: "ZERO_ETIMEOUT", 5: "ZERO_ESTATE"}

EXPORTS = (
    "zero_init_partition", "zero_partition_info", "zero_set_scaler", "zero_step",
    "zero_gather_bucket", "zero_reduce_scatter_bucket", "zero_get_status",
    "zero_bytes_moved", "zero_last_error", "zero_destroy", "zero_step_noalloc",
    "zero_reduce_scatter_bucket_replicas", "zero_quantize_blocks", "zero_dequantize_blocks",
    "zero_gather_bucket_q8", "zero_reduce_scatter_bucket_q", "zero_debug_hold_staged",
    "zero_noalloc_scratch_bytes", "zero_set_persistent", "zero_reduce_scatter_gather_bucket",
)
ZERO_Q_BLOCK = 256


class ZeroError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class Hyper(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float),
                ("max_norm", C.c_float), ("mode", C.c_int32)]


class Result(C.Structure):
    _fields_ = [("overflow", C.c_int32), ("applied", C.c_int32), ("state_slot", C.c_int32),
                ("error", C.c_int32), ("grad_norm", C.c_double), ("clip_coef", C.c_double),
                ("loss_scale", C.c_float), ("reserved", C.c_float),
                ("steps_applied", C.c_int64), ("steps_skipped", C.c_int64)]


class Bytes(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in (
        "psi", "psi_pad", "shard", "n_ranks", "stage", "model_state_bytes_per_rank",
        "comm_elems_paper", "comm_elems_ring", "hbm_read_bytes", "hbm_write_bytes",
        "hbm_read_total", "hbm_write_total")]


_lib = None


def library_path() -> str:
    """libzero_gb300.so to load: $ZERO_GB300_LIB if set, else the in-tree build."""
    return os.environ.get("ZERO_GB300_LIB", LIB_PATH)


def load_library():
    """Load libzero_gb300.so; raise loudly if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ZeroError(3, f"{path} is missing: build it with "
                           "`python -m zero_partitioned_mixed_gb300.build`")
    try:  # make torch's libcudart the one the library binds to, when torch is present
        import torch  # noqa: F401
    except Exception:
        pass
    lib = C.CDLL(path)
    P, U64, I32 = C.c_void_p, C.c_uint64, C.c_int
    lib.zero_init_partition.argtypes = [U64, I32, I32, I32, I32, C.c_uint, C.POINTER(P)]
    lib.zero_partition_info.argtypes = [P, C.POINTER(U64), C.POINTER(U64), C.POINTER(U64), C.POINTER(U64)]
    lib.zero_set_scaler.argtypes = [P, C.c_float, C.c_int64, C.c_int32, P]
    lib.zero_step.argtypes = [P, C.POINTER(P), C.POINTER(P), P, P, P, C.POINTER(Hyper), P]
    lib.zero_gather_bucket.argtypes = [P, U64, U64, P, C.POINTER(P), P]
    lib.zero_reduce_scatter_bucket.argtypes = [P, U64, U64, C.POINTER(P), P, P, P, P, C.POINTER(Hyper), P]
    lib.zero_reduce_scatter_gather_bucket.argtypes = [P, U64, U64, C.POINTER(P), P, P, P, P, C.POINTER(Hyper),
                                                      U64, U64, C.POINTER(P), P]
    lib.zero_reduce_scatter_bucket_replicas.argtypes = [P, U64, U64, C.POINTER(P), P, P, P, C.POINTER(P),
                                                         C.POINTER(Hyper), P]
    lib.zero_quantize_blocks.argtypes = [I32, I32, P, U64, P, P, P]
    lib.zero_dequantize_blocks.argtypes = [I32, I32, P, P, U64, P, P]
    lib.zero_gather_bucket_q8.argtypes = [P, U64, U64, P, C.POINTER(P), C.POINTER(P), P]
    lib.zero_reduce_scatter_bucket_q.argtypes = [P, U64, U64, I32, C.POINTER(P), C.POINTER(P), P, P, P, P,
                                                 C.POINTER(Hyper), P]
    lib.zero_get_status.argtypes = [P, P, C.POINTER(Result)]
    lib.zero_debug_hold_staged.argtypes = [P, C.c_int64]
    lib.zero_bytes_moved.argtypes = [P, C.POINTER(Bytes)]
    lib.zero_set_persistent.argtypes = [P, U64]
    lib.zero_last_error.argtypes = [P]
    lib.zero_last_error.restype = C.c_char_p
    lib.zero_step_noalloc.argtypes = [U64, I32, I32, I32, I32, C.POINTER(P), C.POINTER(P), P, P, P,
                                       C.POINTER(Hyper), C.c_float, C.c_int64, P, P]
    lib.zero_destroy.argtypes = [P]
    lib.zero_destroy.restype = None
    lib.zero_noalloc_scratch_bytes.argtypes = []
    lib.zero_noalloc_scratch_bytes.restype = U64
    for name in EXPORTS:
        if name not in ("zero_last_error", "zero_destroy", "zero_noalloc_scratch_bytes"):
            getattr(lib, name).restype = C.c_int
    _lib = lib
    return lib


def exported_symbols() -> list:
    """Names of the ABI entry points that the loaded library exports."""
    lib = load_library()
    out = []
    for name in EXPORTS:
        try:
            getattr(lib, name)
            out.append(name)
        except AttributeError:
            pass
    return out


# ---------------------------------------------------------------- marshalling
def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs: Optional[Sequence]):
    """A C array of device pointers; an array built earlier passes through."""
    if xs is None:
        return None
    if isinstance(xs, C.Array):
        return xs
    arr = (C.c_void_p * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def pointer_array(tensors: Sequence):
    """The C array of the tensors' device pointers, for calls that are made
    again and again with the same rows: every call that takes a list of
    tensors also takes this array, and skips converting the list.  The
    tensors must stay alive, and in place, while the array is in use."""
    return _ptr_array(list(tensors))


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(rc: int, h) -> None:
    if rc != 0:
        msg = load_library().zero_last_error(h)
        raise ZeroError(rc, msg.decode() if msg else "")


def hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, max_norm=0.0,
          mode=ZERO_MODE_AUTO) -> Hyper:
    return Hyper(lr, beta1, beta2, eps, weight_decay, max_norm, mode)


# ---------------------------------------------------------------- C calls
def zero_init_partition(psi: int, n_ranks: int, stage: int, dtype: int, align: int = 8,
                        flags: int = 0) -> int:
    lib = load_library()
    h = C.c_void_p()
    rc = lib.zero_init_partition(psi, n_ranks, stage, dtype, align, flags, C.byref(h))
    _check(rc, None)
    return h.value


def zero_partition_info(h):
    lib = load_library()
    pp, sh = C.c_uint64(), C.c_uint64()
    n = zero_bytes_moved(h)["n_ranks"]
    offs, real = (C.c_uint64 * n)(), (C.c_uint64 * n)()
    _check(lib.zero_partition_info(h, C.byref(pp), C.byref(sh), offs, real), h)
    return pp.value, sh.value, list(offs), list(real)


def zero_set_scaler(h, loss_scale: float, steps_applied: int = 0, state_slot: int = 0, stream=None):
    _check(load_library().zero_set_scaler(h, loss_scale, steps_applied, state_slot, _stream(stream)), h)


def zero_step(h, grads, params, master, m, v, hyp: Hyper, stream=None):
    lib = load_library()
    rc = lib.zero_step(h, _ptr_array(grads), _ptr_array(params), _ptr(master), _ptr(m), _ptr(v),
                       C.byref(hyp), _stream(stream))
    _check(rc, h)


def zero_gather_bucket(h, a: int, b: int, shard16, out, stream=None):
    rc = load_library().zero_gather_bucket(h, a, b, _ptr(shard16), _ptr_array(out), _stream(stream))
    _check(rc, h)


def zero_reduce_scatter_bucket(h, a: int, b: int, grads, master, m, v, shard16, hyp: Hyper, stream=None):
    rc = load_library().zero_reduce_scatter_bucket(h, a, b, _ptr_array(grads), _ptr(master), _ptr(m),
                                                   _ptr(v), _ptr(shard16), C.byref(hyp), _stream(stream))
    _check(rc, h)


def zero_reduce_scatter_gather_bucket(h, a: int, b: int, grads, master, m, v, shard16, hyp: Hyper, ga: int,
                                      gb: int, out, stream=None):
    rc = load_library().zero_reduce_scatter_gather_bucket(h, a, b, _ptr_array(grads), _ptr(master), _ptr(m),
                                                          _ptr(v), _ptr(shard16), C.byref(hyp), ga, gb,
                                                          _ptr_array(out), _stream(stream))
    _check(rc, h)


def zero_reduce_scatter_bucket_replicas(h, a: int, b: int, grads, master, m, v, params, hyp: Hyper,
                                        stream=None):
    rc = load_library().zero_reduce_scatter_bucket_replicas(h, a, b, _ptr_array(grads), _ptr(master), _ptr(m),
                                                            _ptr(v), _ptr_array(params), C.byref(hyp),
                                                            _stream(stream))
    _check(rc, h)


def zero_quantize_blocks(dtype: int, bits: int, src16, count: int, codes, scales, stream=None):
    _check(load_library().zero_quantize_blocks(dtype, bits, _ptr(src16), count, _ptr(codes), _ptr(scales),
                                               _stream(stream)), None)


def zero_dequantize_blocks(dtype: int, bits: int, codes, scales, count: int, out16, stream=None):
    _check(load_library().zero_dequantize_blocks(dtype, bits, _ptr(codes), _ptr(scales), count, _ptr(out16),
                                                 _stream(stream)), None)


def zero_gather_bucket_q8(h, a: int, b: int, shard16, codes_out, scales_out, stream=None):
    _check(load_library().zero_gather_bucket_q8(h, a, b, _ptr(shard16), _ptr_array(codes_out),
                                                _ptr_array(scales_out), _stream(stream)), h)


def zero_reduce_scatter_bucket_q(h, a: int, b: int, bits: int, codes, scales, master, m, v, shard16, hyp: Hyper,
                                 stream=None):
    _check(load_library().zero_reduce_scatter_bucket_q(h, a, b, bits, _ptr_array(codes), _ptr_array(scales),
                                                       _ptr(master), _ptr(m), _ptr(v), _ptr(shard16), C.byref(hyp),
                                                       _stream(stream)), h)


def zero_get_status(h, stream=None) -> dict:
    """The last step's status.  ZERO_ETIMEOUT raises ZeroError carrying the
    filled status as ``.result``."""
    r = Result()
    rc = load_library().zero_get_status(h, _stream(stream), C.byref(r))
    out = {f: getattr(r, f) for f, _ in Result._fields_ if f != "reserved"}
    if rc == ZERO_ETIMEOUT:
        msg = load_library().zero_last_error(h)
        err = ZeroError(rc, msg.decode() if msg else "")
        err.result = out
        raise err
    _check(rc, h)
    return out


def zero_debug_hold_staged(h, tile: int) -> None:
    _check(load_library().zero_debug_hold_staged(h, int(tile)), h)


def zero_set_persistent(h, p0: int) -> None:
    _check(load_library().zero_set_persistent(h, int(p0)), h)


def zero_bytes_moved(h) -> dict:
    b = Bytes()
    _check(load_library().zero_bytes_moved(h, C.byref(b)), h)
    return {f: getattr(b, f) for f, _ in Bytes._fields_}


def zero_noalloc_scratch_bytes() -> int:
    """Bytes of the static device array behind zero_step_noalloc (host query)."""
    return int(load_library().zero_noalloc_scratch_bytes())


def zero_step_noalloc(psi: int, n_ranks: int, stage: int, dtype: int, align: int, grads, params,
                      master, m, v, hyp: Hyper, loss_scale: float, steps_applied: int, result, stream=None):
    """Two-pass step with all scratch in the library's static device array (no allocation).

    result: device tensor of at least 56 bytes (8-byte aligned) that receives the
    step's zero_result_t; read it with :func:`result_from_device`.
    """
    rc = load_library().zero_step_noalloc(psi, n_ranks, stage, dtype, align, _ptr_array(grads),
                                          _ptr_array(params), _ptr(master), _ptr(m), _ptr(v), C.byref(hyp),
                                          loss_scale, steps_applied, _ptr(result), _stream(stream))
    _check(rc, None)


def result_from_device(t) -> dict:
    """Decode a zero_result_t written to a device (or host) uint8 tensor."""
    raw = bytes(t.view(-1)[:C.sizeof(Result)].cpu().numpy().tobytes())
    r = Result.from_buffer_copy(raw)
    return {f: getattr(r, f) for f, _ in Result._fields_ if f != "reserved"}


def zero_last_error(h) -> str:
    msg = load_library().zero_last_error(h)
    return msg.decode() if msg else ""


def zero_destroy(h) -> None:
    if h:
        load_library().zero_destroy(h)
