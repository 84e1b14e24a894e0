"""ctypes declarations of libdspark's C ABI (include/dspark.h).

The library is loaded from ``_build/libdspark.so`` inside this package.  If it is missing the
import of an op raises: there is no CPU or PyTorch fallback for any call.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
SZ = ctypes.c_size_t
U64 = ctypes.c_uint64

STATUS = {0: "DSPARK_OK", 1: "DSPARK_ERR_INVALID", 2: "DSPARK_ERR_WORKSPACE",
          3: "DSPARK_ERR_CUDA", 4: "DSPARK_ERR_TIMEOUT", 5: "DSPARK_ERR_UNSUPPORTED"}

# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "dspark_workspace_bytes": (SZ, [I, I, I, I, I, I, I]),
    "dspark_markov_draft": (I, [I, I, I, I, I, F, U64, I, P, P, I, P, I, P, P, P, P, P,
                                P, P, P, P, P, P, P, P, SZ, P]),
    "dspark_rnn_draft": (I, [I, I, I, I, I, F, U64, I, P, P, I, P, P, I, P, P, P, P, P, P,
                             P, P, P, P, P, P, P, P, P, SZ, P]),
    "dspark_markov_draft_noalloc": (I, [I, I, I, I, I, F, U64, I, P, P, P, I, P, P, P, P, P,
                                        P, P, P, P, P, P, P, P, P]),
    "dspark_confidence": (I, [I, I, I, I, I, I, P, P, I, P, P, P, P, P, P]),
    "dspark_tv_label": (I, [I, I, F, P, P, P, P, P]),
    "dspark_prefix_schedule": (I, [I, I, P, P, P, P, P]),
    "dspark_verify_workspace_bytes": (SZ, [I, I, I]),
    "dspark_verify": (I, [I, I, I, F, U64, P, P, P, P, P, P, SZ, P]),
    "dspark_draft_loss_workspace_bytes": (SZ, [I, I, I]),
    "dspark_sts_workspace_bytes": (SZ, [I, I, I, I]),
    "dspark_sts": (I, [I, I, P, P, I, P, I, P, P, P, P, SZ, P]),
    "dspark_draft_loss": (I, [I, I, I, F, P, P, P, P, F, F, F, P, P, P, P, P, SZ, P]),
    "dspark_get_status": (I, [P, SZ, P]),
    "dspark_last_error": (ctypes.c_char_p, []),
    "dspark_draft_path": (I, [I, I, I, I, I]),
    "dspark_draft_launches": (I, [I, I, I, I, I]),
    "dspark_draft_cluster": (I, [I, I, I, I, I]),
    "dspark_draft_loss_launches": (I, [I, I, I, I]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded CDLL.  Raises RuntimeError when the library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libdspark is not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class DsparkError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().dspark_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS.get(code, code)}: {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != 0:
        raise DsparkError(code, where)
