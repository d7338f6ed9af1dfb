"""ctypes binding of the diagnostic library lib/libldn_diag.so
(include/ldn_diag.h), which the tests alone load: the product library
libldn.so does not carry these entry points."""
import ctypes
import os
import threading

from gated_delta_rule_chunkwise_gb300 import build as ldn_build

_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "ldn_diag_umma": ([_P] * 3 + [_I] * 6 + [_P], _I),
    "ldn_diag_umma_tmem_a": ([_P] * 3 + [_I] * 4 + [_P], _I),
    "ldn_diag_tma_sw128": ([_P] * 2 + [_I] * 4 + [_P], _I),
    "ldn_diag_wait_timeout": ([ctypes.c_longlong, _P, _P], _I),
    "ldn_diag_get_device_status": ([_P], _I),
}
_lock = threading.Lock()
_lib = None


def load():
    """Build (if stale) and load libldn_diag.so with its argument types."""
    global _lib
    with _lock:
        if _lib is None:
            ldn_build.build()
            lib = ctypes.CDLL(ldn_build.DIAG_LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def status(stream=None) -> int:
    """Read and clear the diagnostic kernels' status word (after a sync)."""
    return int(load().ldn_diag_get_device_status(stream))
