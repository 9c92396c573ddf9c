"""GB300 (sm_103a) modulation-fused NVFP4 activation producer and block-scaled GEMM.

Python binding of the C-ABI library ``libh3fp4.so`` (see ``include/h3fp4.h``).
The ``h3fp4_*`` functions mirror the C entry points one to one and take raw
device pointers (ints); the short-named helpers below them take torch tensors,
allocate outputs with torch and pass pointers plus torch's current stream.
Every arithmetic step runs in the library's CUDA kernels: there is no CPU or
PyTorch fallback, and every call raises if the library is missing or returns
an error status.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libh3fp4.so")
MAX_SEGMENTS = 16

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_STATUS = ctypes.c_int

# (name, argtypes, restype) of every exported entry point.
_SIGNATURES = {
    "h3fp4_modulate_absmax": ([_P, _I64, _I64, _I64, _P, _P, _I64, _P, _I32, _P, _P, _P], _STATUS),
    "h3fp4_modulate_pack": ([_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _I32, _P, _P, _P, _P], _STATUS),
    "h3fp4_modulate_produce": ([_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _I32, _P, _P, _P, _P, _P], _STATUS),
    "h3fp4_swiglu_pack": ([_P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P], _STATUS),
    "h3fp4_quantize_pack": ([_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P], _STATUS),
    "h3fp4_gemm_gated_residual": ([_P, _P, _P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I64, _P, _I64, _I64, _I64, _I64,
                                   _I64, _P, _P], _STATUS),
    "h3fp4_gemm": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P], _STATUS),
    "h3fp4_swizzle_scales": ([_P, _I64, _I64, _I64, _P, _P], _STATUS),
    "h3fp4_swiglu_pack_noalloc": ([_P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P], _STATUS),
    "h3fp4_device_error": ([_P], _STATUS),
    "h3fp4_diag_producer_barrier_timeout": ([_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, ctypes.c_uint32, _P],
                                            _STATUS),
    "h3fp4_diag_gemm_wait_timeout": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, ctypes.c_uint32, _P],
                                     _STATUS),
    "h3fp4_status_string": ([_STATUS], ctypes.c_char_p),
    "h3fp4_build_info": ([], ctypes.c_char_p),
}

STATUS_NAMES = {0: "H3FP4_OK", 1: "H3FP4_ERR_NULL", 2: "H3FP4_ERR_ALIGN", 3: "H3FP4_ERR_SHAPE",
                4: "H3FP4_ERR_UNSUPPORTED", 5: "H3FP4_ERR_CUDA", 6: "H3FP4_ERR_DEVICE"}


class H3FP4Error(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {STATUS_NAMES.get(status, status)} ({_status_text(status)})")


class GemmConfig(ctypes.Structure):
    _fields_ = [("n_group", _I32), ("stages", _I32), ("cta_pair", _I32), ("reserved", _I32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _status_text(status: int) -> str:
    try:
        return lib().h3fp4_status_string(status).decode()
    except Exception:  # library not loadable: fall back to the enum name
        return STATUS_NAMES.get(status, "unknown")


def _call(name: str, *args) -> None:
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise H3FP4Error(name, st)


def _offsets(seg_row_offsets):
    arr = (ctypes.c_int32 * len(seg_row_offsets))(*[int(v) for v in seg_row_offsets])
    return arr, len(seg_row_offsets) - 1


# ----------------------------------------------------------------------------
# Raw C-ABI mirrors: device pointers as ints, stream as an int handle (0 = default).
# ----------------------------------------------------------------------------
def h3fp4_modulate_absmax(x, ldx, m, d, shift, scale, ld_mod, seg_row_offsets, tensor_scale, scratch, stream=0):
    offs, nseg = _offsets(seg_row_offsets)
    _call("h3fp4_modulate_absmax", x, ldx, m, d, shift, scale, ld_mod, offs, nseg, tensor_scale, scratch, stream)


def h3fp4_modulate_pack(x, ldx, m, m_pad, d, shift, scale, ld_mod, seg_row_offsets, tensor_scale, qdata, sfa,
                        stream=0):
    offs, nseg = _offsets(seg_row_offsets)
    _call("h3fp4_modulate_pack", x, ldx, m, m_pad, d, shift, scale, ld_mod, offs, nseg, tensor_scale, qdata, sfa,
          stream)


def h3fp4_modulate_produce(x, ldx, m, m_pad, d, shift, scale, ld_mod, seg_row_offsets, tensor_scale, scratch, qdata,
                           sfa, stream=0):
    offs, nseg = _offsets(seg_row_offsets)
    _call("h3fp4_modulate_produce", x, ldx, m, m_pad, d, shift, scale, ld_mod, offs, nseg, tensor_scale, scratch,
          qdata, sfa, stream)


def h3fp4_swiglu_pack(gate, ldg, up, ldu, m, m_pad, f, tensor_scale, scratch, qdata, sfa, h_workspace=None,
                      stream=0):
    _call("h3fp4_swiglu_pack", gate, ldg, up, ldu, m, m_pad, f, tensor_scale, scratch, qdata, sfa, h_workspace,
          stream)


def h3fp4_quantize_pack(x, ldx, m, m_pad, d, tensor_scale, scratch, qdata, sfa, stream=0):
    _call("h3fp4_quantize_pack", x, ldx, m, m_pad, d, tensor_scale, scratch, qdata, sfa, stream)


def h3fp4_gemm(a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k, cfg: GemmConfig | None = None, stream=0):
    _call("h3fp4_gemm", a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k,
          ctypes.byref(cfg) if cfg is not None else None, stream)


def h3fp4_gemm_gated_residual(a_q, a_sf, a_ts, b_q, b_sf, b_ts, gate, ld_gate, seg_row_offsets, residual, ldr, out,
                              ldo, m, m_pad, n, k, cfg: GemmConfig | None = None, stream=0):
    offs, nseg = _offsets(seg_row_offsets)
    _call("h3fp4_gemm_gated_residual", a_q, a_sf, a_ts, b_q, b_sf, b_ts, gate, ld_gate, offs, nseg, residual, ldr,
          out, ldo, m, m_pad, n, k, ctypes.byref(cfg) if cfg is not None else None, stream)


def h3fp4_swizzle_scales(sf_logical, rows, cols, ld, sf_out, stream=0):
    _call("h3fp4_swizzle_scales", sf_logical, rows, cols, ld, sf_out, stream)


def h3fp4_swiglu_pack_noalloc(gate, ldg, up, ldu, m, m_pad, f, tensor_scale, qdata, sfa, stream=0):
    """The SwiGLU producer with library-owned static scratch, for callers that cannot allocate."""
    _call("h3fp4_swiglu_pack_noalloc", gate, ldg, up, ldu, m, m_pad, f, tensor_scale, qdata, sfa, stream)


NOALLOC_MAX_ELEMENTS = 1 << 22


def h3fp4_device_error() -> int:
    code = ctypes.c_uint32(0)
    _call("h3fp4_device_error", ctypes.byref(code))
    return code.value


def h3fp4_diag_producer_barrier_timeout(x, ldx, m, m_pad, d, tensor_scale, scratch, qdata, sfa, limit_us, stream=0):
    """Failure-detection check: the cooperative producer's grid barrier gives up after limit_us."""
    _call("h3fp4_diag_producer_barrier_timeout", x, ldx, m, m_pad, d, tensor_scale, scratch, qdata, sfa, limit_us,
          stream)


def h3fp4_diag_gemm_wait_timeout(a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k, limit_us, stream=0):
    """Failure-detection check: the default GEMM with its loads withheld; its waits give up after limit_us."""
    _call("h3fp4_diag_gemm_wait_timeout", a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k, limit_us, stream)


def h3fp4_build_info() -> str:
    return lib().h3fp4_build_info().decode()


# ----------------------------------------------------------------------------
# torch-tensor helpers (allocation with torch, pointers + current stream to the C ABI)
# ----------------------------------------------------------------------------
def sf_rows(rows: int) -> int:
    """Rows of a scale buffer: rows rounded up to a multiple of 128."""
    return -(-rows // 128) * 128


def sf_bytes(rows: int, width: int) -> int:
    return sf_rows(rows) * (width // 16)


def _stream(stream):
    import torch
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def modulate_absmax(x, shift, scale, seg_row_offsets, *, tensor_scale=None, scratch=None, stream=None):
    """Pass 1: returns the FP32 tensor scale (1-element device tensor)."""
    import torch
    _need_cuda(x, shift, scale)
    m, d = x.shape
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=x.device)
    if scratch is None:
        scratch = torch.empty(2, dtype=torch.int32, device=x.device)
    h3fp4_modulate_absmax(x.data_ptr(), x.stride(0), m, d, shift.data_ptr(), scale.data_ptr(), shift.stride(0),
                          seg_row_offsets, tensor_scale.data_ptr(), scratch.data_ptr(), _stream(stream))
    return tensor_scale


def modulate_pack(x, shift, scale, seg_row_offsets, tensor_scale, m_pad, *, qdata=None, sfa=None, stream=None):
    """Pass 2: returns (qdata [m_pad, d/2] uint8, sfa flat uint8 in the scale layout)."""
    import torch
    _need_cuda(x, shift, scale, tensor_scale)
    m, d = x.shape
    if qdata is None:
        qdata = torch.empty(m_pad, d // 2, dtype=torch.uint8, device=x.device)
    if sfa is None:
        sfa = torch.empty(sf_bytes(m_pad, d), dtype=torch.uint8, device=x.device)
    h3fp4_modulate_pack(x.data_ptr(), x.stride(0), m, m_pad, d, shift.data_ptr(), scale.data_ptr(), shift.stride(0),
                        seg_row_offsets, tensor_scale.data_ptr(), qdata.data_ptr(), sfa.data_ptr(), _stream(stream))
    return qdata, sfa


def modulate_produce(x, shift, scale, seg_row_offsets, m_pad, *, tensor_scale=None, scratch=None, qdata=None,
                     sfa=None, stream=None):
    """Both modulation-producer passes in one launch: returns (tensor_scale, qdata, sfa)."""
    import torch
    _need_cuda(x, shift, scale)
    m, d = x.shape
    dev = x.device
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = torch.empty(2, dtype=torch.int32, device=dev)
    if qdata is None:
        qdata = torch.empty(m_pad, d // 2, dtype=torch.uint8, device=dev)
    if sfa is None:
        sfa = torch.empty(sf_bytes(m_pad, d), dtype=torch.uint8, device=dev)
    h3fp4_modulate_produce(x.data_ptr(), x.stride(0), m, m_pad, d, shift.data_ptr(), scale.data_ptr(),
                           shift.stride(0), seg_row_offsets, tensor_scale.data_ptr(), scratch.data_ptr(),
                           qdata.data_ptr(), sfa.data_ptr(), _stream(stream))
    return tensor_scale, qdata, sfa


def swiglu_pack(gate, up, m_pad, *, h_workspace=None, tensor_scale=None, scratch=None, qdata=None, sfa=None,
                stream=None):
    """SwiGLU producer: returns (tensor_scale, qdata, sfa)."""
    import torch
    _need_cuda(gate, up, h_workspace)
    m, f = gate.shape
    dev = gate.device
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = torch.empty(2, dtype=torch.int32, device=dev)
    if qdata is None:
        qdata = torch.empty(m_pad, f // 2, dtype=torch.uint8, device=dev)
    if sfa is None:
        sfa = torch.empty(sf_bytes(m_pad, f), dtype=torch.uint8, device=dev)
    h3fp4_swiglu_pack(gate.data_ptr(), gate.stride(0), up.data_ptr(), up.stride(0), m, m_pad, f,
                      tensor_scale.data_ptr(), scratch.data_ptr(), qdata.data_ptr(), sfa.data_ptr(),
                      h_workspace.data_ptr() if h_workspace is not None else None, _stream(stream))
    return tensor_scale, qdata, sfa


def quantize_pack(x, m_pad, *, tensor_scale=None, scratch=None, qdata=None, sfa=None, stream=None):
    """NVFP4 producer of a plain bf16 activation (both passes): returns (tensor_scale, qdata, sfa)."""
    import torch
    _need_cuda(x)
    m, d = x.shape
    dev = x.device
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = torch.empty(2, dtype=torch.int32, device=dev)
    if qdata is None:
        qdata = torch.empty(m_pad, d // 2, dtype=torch.uint8, device=dev)
    if sfa is None:
        sfa = torch.empty(sf_bytes(m_pad, d), dtype=torch.uint8, device=dev)
    h3fp4_quantize_pack(x.data_ptr(), x.stride(0), m, m_pad, d, tensor_scale.data_ptr(), scratch.data_ptr(),
                        qdata.data_ptr(), sfa.data_ptr(), _stream(stream))
    return tensor_scale, qdata, sfa


def gemm(a_q, a_sf, a_ts, b_q, b_sf, b_ts, m, *, out=None, cfg: GemmConfig | None = None, stream=None):
    """C[m, n] bf16 (returned as int16 patterns unless `out` is given)."""
    import torch
    _need_cuda(a_q, a_sf, a_ts, b_q, b_sf, b_ts, out)
    m_pad, kh = a_q.shape
    n = b_q.shape[0]
    if out is None:
        out = torch.empty(m, n, dtype=torch.int16, device=a_q.device)
    h3fp4_gemm(a_q.data_ptr(), a_sf.data_ptr(), a_ts.data_ptr(), b_q.data_ptr(), b_sf.data_ptr(), b_ts.data_ptr(),
               out.data_ptr(), out.stride(0), m, m_pad, n, 2 * kh, cfg, _stream(stream))
    return out


def gemm_gated_residual(a_q, a_sf, a_ts, b_q, b_sf, b_ts, m, gate, seg_row_offsets, residual, *, out=None,
                       cfg: GemmConfig | None = None, stream=None):
    """out = RN_bf16(residual + RN_bf16(gate_s * C)) with C the GEMM result; pass
    out=residual to update the residual in place.  Returns out (int16 bf16 patterns)."""
    import torch
    _need_cuda(a_q, a_sf, a_ts, b_q, b_sf, b_ts, gate, residual, out)
    m_pad, kh = a_q.shape
    n = b_q.shape[0]
    if out is None:
        out = torch.empty(m, n, dtype=torch.int16, device=a_q.device)
    h3fp4_gemm_gated_residual(a_q.data_ptr(), a_sf.data_ptr(), a_ts.data_ptr(), b_q.data_ptr(), b_sf.data_ptr(),
                              b_ts.data_ptr(), gate.data_ptr(), gate.stride(0), seg_row_offsets,
                              residual.data_ptr(), residual.stride(0), out.data_ptr(), out.stride(0), m, m_pad, n,
                              2 * kh, cfg, _stream(stream))
    return out


def swizzle_scales(sf_logical, *, out=None, stream=None):
    """Logical [rows, cols] uint8 scales -> flat scale-layout bytes (rows padded to 128)."""
    import torch
    _need_cuda(sf_logical, out)
    rows, cols = sf_logical.shape
    if out is None:
        out = torch.empty(sf_rows(rows) * cols, dtype=torch.uint8, device=sf_logical.device)
    h3fp4_swizzle_scales(sf_logical.data_ptr(), rows, cols, sf_logical.stride(0), out.data_ptr(), _stream(stream))
    return out
