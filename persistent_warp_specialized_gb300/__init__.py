"""Python binding of libtg, the persistent warp-specialized GEMM for GB300 (sm_103a).

Argument marshalling only: every function here forwards to the C entry point of the same
name declared in ``include/tg.h``; all of the GEMM and the tile scheduling run in the
library's CUDA kernels.  Tensors are passed by their device pointers (``data_ptr()``);
PyTorch only provides device memory and streams.  There is no fallback: if ``libtg.so``
is missing or fails to load, every call raises.

Build the library with ``persistent_warp_specialized_gb300._build.build()`` (nvcc, sm_103a).
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtg.so")

TG_F16 = 0
TG_BF16 = 1
TG_OK = 0
TG_ERR_ARG = -1
TG_ERR_ALIGN = -2
TG_ERR_CUDA = -3
TG_ERR_TIMEOUT = -4
TG_VARIANT_AUTO = 0
TG_VARIANT_SINGLE = 1
TG_VARIANT_PAIR = 2
TG_VARIANT_PAIR_WIDE = 3
TG_SCHEDULE_PLAIN = 0x100
TG_SCHEDULE_COLUMN_MAJOR = 0x200
TG_SCHEDULE_SPLIT_TAIL = 0x1
TG_SCHEDULE_DYNAMIC = 0x400
TG_EPILOGUE_DIRECT = 0x800
TG_SHAPE_MXFP8 = 0x1000
TG_SCHEDULE_STREAMK = 0x2000
TG_SHAPE_WORKSPACE = 0x4000
TG_SCHEDULE_NOALLOC_MAX_UNITS = 65536   # scratch rows of tg_tile_schedule_noalloc
VARIANTS = {"auto": TG_VARIANT_AUTO, "single": TG_VARIANT_SINGLE, "pair": TG_VARIANT_PAIR,
            "wide": TG_VARIANT_PAIR_WIDE}

DTYPES = {"f16": TG_F16, "bf16": TG_BF16}

EXPORTED = (
    "tg_gemm_persistent",
    "tg_gemm_persistent_ex",
    "tg_gemm_persistent_ws",
    "tg_gemm_workspace_bytes",
    "tg_tile_schedule",
    "tg_tile_schedule_ex",
    "tg_tile_schedule_noalloc",
    "tg_last_error",
    "tg_gemm_config",
    "tg_gemm_launch_shape",
    "tg_gemm_persistent_debug",
    "tg_device_status",
    "tg_gemm_persistent_host",
    "tg_gemm_mxfp8",
    "tg_gemm_mxfp8_ex",
    "tg_gemm_mxfp8_debug",
    "tg_mxfp8_scale_bytes",
    "tg_mxfp8_pack_scales",
)


class TgError(RuntimeError):
    def __init__(self, code, message):
        super().__init__(f"tg error {code}: {message}")
        self.code = code


_lib = None


def load_library(path=LIB_PATH):
    """Load libtg.so (once) and declare its C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built; run persistent_warp_specialized_gb300._build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
    lib.tg_gemm_persistent.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
    lib.tg_gemm_persistent.restype = i32
    lib.tg_gemm_persistent_ex.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, i32]
    lib.tg_gemm_persistent_ex.restype = i32
    lib.tg_gemm_persistent_ws.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, i32, vp, i64]
    lib.tg_gemm_persistent_ws.restype = i32
    lib.tg_gemm_workspace_bytes.argtypes = [i64, i64, i64, i32]
    lib.tg_gemm_workspace_bytes.restype = i64
    lib.tg_tile_schedule.argtypes = [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.tg_tile_schedule.restype = i32
    lib.tg_tile_schedule_ex.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.tg_tile_schedule_ex.restype = i32
    lib.tg_tile_schedule_noalloc.argtypes = [i32, i32, i32, i32, i32,
                                             ctypes.POINTER(ctypes.c_int32)]
    lib.tg_tile_schedule_noalloc.restype = i32
    lib.tg_last_error.argtypes = []
    lib.tg_last_error.restype = ctypes.c_char_p
    ip = ctypes.POINTER(ctypes.c_int)
    lib.tg_gemm_config.argtypes = [ip, ip, ip, ip, ip]
    lib.tg_gemm_config.restype = i32
    lib.tg_gemm_launch_shape.argtypes = [i64, i64, i64, i32] + [ip] * 12 + [
        ctypes.POINTER(ctypes.c_int64)]
    lib.tg_gemm_launch_shape.restype = i32
    lib.tg_gemm_persistent_debug.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, i32, vp, u64,
                                             i64, vp, i64]
    lib.tg_gemm_persistent_debug.restype = i32
    lib.tg_device_status.argtypes = [vp]
    lib.tg_device_status.restype = i32
    lib.tg_gemm_persistent_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.tg_gemm_persistent_host.restype = i32
    lib.tg_gemm_mxfp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.tg_gemm_mxfp8.restype = i32
    lib.tg_gemm_mxfp8_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, i32]
    lib.tg_gemm_mxfp8_ex.restype = i32
    lib.tg_gemm_mxfp8_debug.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, i32, vp, u64,
                                        i64]
    lib.tg_gemm_mxfp8_debug.restype = i32
    lib.tg_mxfp8_scale_bytes.argtypes = [i64, i64]
    lib.tg_mxfp8_scale_bytes.restype = i64
    lib.tg_mxfp8_pack_scales.argtypes = [vp, vp, i64, i64, vp]
    lib.tg_mxfp8_pack_scales.restype = i32
    _lib = lib
    return lib


def _check(rc):
    if rc < 0:
        raise TgError(rc, load_library().tg_last_error().decode(errors="replace"))
    return rc


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):          # numpy array (host memory)
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x).__name__}")


def _dtype(d):
    return DTYPES[d] if isinstance(d, str) else int(d)


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def tg_last_error():
    return load_library().tg_last_error().decode(errors="replace")


def tg_gemm_persistent(A, B, C, M, N, K, dtype, stream=None):
    """C = A . B (device buffers; asynchronous on ``stream``, default: torch's current)."""
    return _check(load_library().tg_gemm_persistent(
        _ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype(dtype), _stream(stream)))


def _group(g):
    """TG_SCHEDULE_GROUP(g): the grouped order's width (None: the library's default, 8)."""
    if g is None:
        return 0
    if not 1 <= int(g) <= 255:
        raise ValueError(f"group width {g} outside 1..255")
    return int(g) << 16


def _variant(v, plain=False, column_major=False, dynamic=False, group=None, direct=False,
             streamk=False):
    """"auto" / "single" / "pair" / "wide" (or a TG_VARIANT_* int) plus the schedule flags."""
    code = VARIANTS[v] if isinstance(v, str) else int(v)
    return (code | (TG_SCHEDULE_PLAIN if plain else 0)
            | (TG_SCHEDULE_COLUMN_MAJOR if column_major else 0)
            | (TG_SCHEDULE_DYNAMIC if dynamic else 0) | _group(group)
            | (TG_EPILOGUE_DIRECT if direct else 0)
            | (TG_SCHEDULE_STREAMK if streamk else 0))


def _nbytes(ws, workspace_bytes):
    if ws is None:
        return 0
    if workspace_bytes is not None:
        return int(workspace_bytes)
    if hasattr(ws, "numel") and hasattr(ws, "element_size"):
        return ws.numel() * ws.element_size()
    raise ValueError("workspace_bytes is needed for a raw workspace pointer")


def tg_gemm_persistent_ex(A, B, C, M, N, K, dtype, stream=None, variant="auto", plain=False,
                          column_major=False, dynamic=False, group=None, direct=False):
    """tg_gemm_persistent with an explicit kernel variant ("auto", "single", "pair", "wide");
    ``plain`` walks the page's tile order with no tail split; ``column_major`` the scheduler's
    column-major order."""
    return _check(load_library().tg_gemm_persistent_ex(
        _ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype(dtype), _stream(stream),
        _variant(variant, plain, column_major, dynamic, group, direct)))


def tg_gemm_persistent_ws(A, B, C, M, N, K, dtype, workspace, stream=None, variant="auto",
                          plain=False, column_major=False, group=None, streamk=False,
                          workspace_bytes=None):
    """tg_gemm_persistent_ex with a workspace (a CUDA tensor of at least tg_gemm_workspace_bytes
    bytes, or None); with ``streamk`` the CTA-pair kernels split the last partial wave of tiles
    along K (the stream-K tail) whenever there is one."""
    return _check(load_library().tg_gemm_persistent_ws(
        _ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype(dtype), _stream(stream),
        _variant(variant, plain, column_major, False, group, False, streamk), _ptr(workspace),
        _nbytes(workspace, workspace_bytes)))


def tg_gemm_workspace_bytes(M, N, K, variant="auto", plain=False, column_major=False,
                            group=None, streamk=False):
    """Workspace bytes tg_gemm_persistent_ws needs on the current device (0: none)."""
    n = load_library().tg_gemm_workspace_bytes(
        M, N, K, _variant(variant, plain, column_major, False, group, False, streamk))
    return _check(n) if n < 0 else n


def tg_gemm_persistent_debug(A, B, C, M, N, K, dtype, stream=None, variant="auto", trace=None,
                             watchdog_ns=0, inject_skip_phase=-1, plain=False,
                             column_major=False, dynamic=False, group=None, workspace=None,
                             streamk=False, workspace_bytes=None):
    return _check(load_library().tg_gemm_persistent_debug(
        _ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype(dtype), _stream(stream),
        _variant(variant, plain, column_major, dynamic, group, False, streamk), _ptr(trace),
        watchdog_ns, inject_skip_phase, _ptr(workspace), _nbytes(workspace, workspace_bytes)))


def tg_gemm_persistent_host(A_host, B_host, C_host, A_dev, B_dev, C_dev, M, N, K, dtype,
                            stream=None):
    return _check(load_library().tg_gemm_persistent_host(
        _ptr(A_host), _ptr(B_host), _ptr(C_host), _ptr(A_dev), _ptr(B_dev), _ptr(C_dev),
        M, N, K, _dtype(dtype), _stream(stream)))


def tg_device_status(stream=None):
    return _check(load_library().tg_device_status(_stream(stream)))


def tg_gemm_config():
    vals = [ctypes.c_int() for _ in range(5)]
    _check(load_library().tg_gemm_config(*[ctypes.byref(v) for v in vals]))
    keys = ("block_m", "block_n", "block_k", "stages", "group")
    return dict(zip(keys, (v.value for v in vals)))


def tg_gemm_launch_shape(M, N, K, variant="auto", plain=False, dynamic=False,
                         column_major=False, group=None, mxfp8=False, workspace=False,
                         streamk=False):
    """The persistent launch (and traversal) the library uses for M x N x K on the current
    device: of the dense GEMM, or with ``mxfp8`` of the block-scaled MXFP8 GEMM; with
    ``workspace`` the launch of tg_gemm_persistent_ws (with ``streamk``: the stream-K tail)."""
    vals = [ctypes.c_int() for _ in range(12)]
    ws = ctypes.c_int64()
    code = (_variant(variant, plain, column_major, dynamic, group, False, streamk)
            | (TG_SHAPE_MXFP8 if mxfp8 else 0) | (TG_SHAPE_WORKSPACE if workspace else 0))
    _check(load_library().tg_gemm_launch_shape(M, N, K, code, *[ctypes.byref(v) for v in vals],
                                               ctypes.byref(ws)))
    keys = ("variant", "tile_m", "tile_n", "m_tiles", "n_tiles", "workers", "ctas",
            "split_from", "units", "group", "column_major", "sk_tiles")
    out = dict(zip(keys, (v.value for v in vals)))
    out["workspace_bytes"] = ws.value
    return out


def tg_tile_schedule(m_blocks, n_blocks, num_sms, group):
    """Rows (worker, w, bx, by) of the device scheduler, as a list of 4-tuples."""
    rows = max(0, m_blocks) * max(0, n_blocks)
    buf = (ctypes.c_int32 * (4 * max(rows, 1)))()
    n = _check(load_library().tg_tile_schedule(m_blocks, n_blocks, num_sms, group, buf))
    return [tuple(buf[4 * i: 4 * i + 4]) for i in range(n)]


def tg_tile_schedule_ex(m_blocks, n_blocks, num_sms, group, split_tail=True, column_major=False):
    """Rows (worker, w, bx, by, part) of the device scheduler over work units."""
    rows = 2 * max(0, m_blocks) * max(0, n_blocks)
    buf = (ctypes.c_int32 * (5 * max(rows, 1)))()
    flags = (TG_SCHEDULE_SPLIT_TAIL if split_tail else 0) | (
        TG_SCHEDULE_COLUMN_MAJOR if column_major else 0)
    n = _check(load_library().tg_tile_schedule_ex(m_blocks, n_blocks, num_sms, group, flags, buf))
    return [tuple(buf[5 * i: 5 * i + 5]) for i in range(n)]


def tg_tile_schedule_noalloc(m_blocks, n_blocks, num_sms, group, split_tail=True,
                             column_major=False):
    """The rows of tg_tile_schedule_ex, from the entry point that allocates no device memory
    (for callers whose device memory is all owned by their own allocator, or that must not
    stall on cudaFree).  At most TG_SCHEDULE_NOALLOC_MAX_UNITS units."""
    rows = min(2 * max(0, m_blocks) * max(0, n_blocks), TG_SCHEDULE_NOALLOC_MAX_UNITS)
    buf = (ctypes.c_int32 * (5 * max(rows, 1)))()
    flags = (TG_SCHEDULE_SPLIT_TAIL if split_tail else 0) | (
        TG_SCHEDULE_COLUMN_MAJOR if column_major else 0)
    n = _check(load_library().tg_tile_schedule_noalloc(m_blocks, n_blocks, num_sms, group, flags,
                                                       buf))
    return [tuple(buf[5 * i: 5 * i + 5]) for i in range(n)]


def _mx_flags(variant="auto", plain=False, column_major=False, group=None):
    return _variant(variant, plain, column_major, False, group)


def tg_mxfp8_scale_bytes(rows, K):
    return _check(load_library().tg_mxfp8_scale_bytes(rows, K))


def tg_mxfp8_pack_scales(sf, packed, rows, K, stream=None):
    return _check(load_library().tg_mxfp8_pack_scales(_ptr(sf), _ptr(packed), rows, K,
                                                      _stream(stream)))


def mxfp8_pack(sf, K, stream=None):
    """torch convenience: packed scales of a CUDA uint8 tensor sf [rows, K/32] (a new tensor)."""
    import torch

    rows = sf.shape[0]
    out = torch.empty(tg_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device=sf.device)
    tg_mxfp8_pack_scales(sf, out, rows, K, stream)
    return out


def tg_gemm_mxfp8(A, SFA, B, SFB, C, M, N, K, out_dtype="bf16", stream=None):
    """Block-scaled MXFP8 GEMM: A [M, K], B [N, K] E4M3 bytes; SFA, SFB their packed E8M0
    scales (tg_mxfp8_pack_scales); C [M, N] in ``out_dtype``."""
    return _check(load_library().tg_gemm_mxfp8(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _dtype(out_dtype),
        _stream(stream)))


def tg_gemm_mxfp8_ex(A, SFA, B, SFB, C, M, N, K, out_dtype="bf16", stream=None, variant="auto",
                     plain=False, column_major=False, group=None):
    return _check(load_library().tg_gemm_mxfp8_ex(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _dtype(out_dtype),
        _stream(stream), _mx_flags(variant, plain, column_major, group)))


def tg_gemm_mxfp8_debug(A, SFA, B, SFB, C, M, N, K, out_dtype="bf16", stream=None, trace=None,
                        watchdog_ns=0, inject_skip_phase=-1, variant="auto", plain=False,
                        column_major=False, group=None):
    return _check(load_library().tg_gemm_mxfp8_debug(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _dtype(out_dtype),
        _stream(stream), _mx_flags(variant, plain, column_major, group), _ptr(trace), watchdog_ns,
        inject_skip_phase))


def gemm(a, b, out=None, stream=None):
    """torch convenience: C = a @ b for contiguous 2-D fp16/bf16 CUDA tensors."""
    import torch

    names = {torch.float16: "f16", torch.bfloat16: "bf16"}
    if a.dtype != b.dtype or a.dtype not in names:
        raise TypeError("a and b must both be float16 or both bfloat16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shapes {tuple(a.shape)} and {tuple(b.shape)} do not contract")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous row-major")
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=a.dtype, device=a.device)
    tg_gemm_persistent(a, b, out, M, N, K, names[a.dtype], stream)
    return out


def mxfp8_gemm(a, sa, b, sb, out=None, out_dtype="bf16", stream=None):
    """torch convenience: the block-scaled MXFP8 product of CUDA uint8 tensors a [M, K] and
    b [N, K] (E4M3) with row-major E8M0 scales sa [M, K/32] and sb [N, K/32]; packs the scales
    (tg_mxfp8_pack_scales) and runs tg_gemm_mxfp8 into ``out`` (a new [M, N] tensor if None)."""
    import torch

    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K or tuple(sa.shape) != (M, K // 32) or tuple(sb.shape) != (N, K // 32):
        raise ValueError("shapes: a [M, K], b [N, K], sa [M, K/32], sb [N, K/32]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float16,
                          device=a.device)
    tg_gemm_mxfp8(a, mxfp8_pack(sa, K, stream), b, mxfp8_pack(sb, K, stream), out, M, N, K,
                  out_dtype, stream)
    return out
